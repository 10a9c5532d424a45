#!/usr/bin/env python3
"""Benchmark of the batched acceptance step (libsdcp on GB300).

One step = one sdcp_verify_batch call over one synthetic verify batch (all phases:
row statistics of the sampling profile, acceptance tests, first-rejection scan, draw of
the additional token).  Default workload: B=64 sessions, M=8, V=32000, bf16 logits,
speculative sampling at T=0.7 with top_k=50.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  value = verified tokens/s (sum of n_out over the batch,
summed over ranks, divided by the max over ranks of the mean device time of a step;
inputs resident in HBM; L2 flushed by a 256 MiB write between timed steps).
N > 1 runs under torchrun, one process per GPU, each with its own batch (weak scaling;
the sessions of different GPUs are independent, no collective on the data path).
--impl reference times the CPU oracle (oracle/, fp64 C) on the host cores instead.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified tokens/sec and achieved HBM GB/s (% of GB300 peak) per verify batch"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "topk50"
L2_FLUSH_BYTES = 256 << 20
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
KERNEL_SOURCES = ["speculative_decoding_verification_sdcp_gb300/csrc/sdcp_rows.cu",
                  "speculative_decoding_verification_sdcp_gb300/csrc/sdcp_session.cuh",
                  "speculative_decoding_verification_sdcp_gb300/csrc/sdcp_device.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sessions", type=int, default=None,
                    help="keep only the first N sessions of the workload (small cases for ncu)")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------
# distributed plumbing (torchrun): barrier and max/sum over ranks
# ------------------------------------------------------------------------------------------
class Dist:
    def __init__(self, want_gpus: int):
        import torch
        self.torch = torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist
        if want_gpus != self.world and self.rank == 0 and self.world > 1:
            print("warning: --gpus %d but WORLD_SIZE %d" % (want_gpus, self.world), file=sys.stderr)

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def reduce(self, value: float, op: str) -> float:
        if not self.pg:
            return value
        t = self.torch.tensor([value], dtype=self.torch.float64,
                              device="cuda" if self.torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX if op == "max" else self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + CLOCK_QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the row kernel from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "row_stats_kernel_%s.md" % workload)
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", txt)
    if not m or not t or m.group(1) != kernel_hash():
        return None
    return int(t.group(1))


# ------------------------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# ------------------------------------------------------------------------------------------
def oracle_sessions(batch, sessions):
    """Host arrays of the given sessions, re-laid out as a batch of their own."""
    import numpy as np
    import torch
    from speculative_decoding_verification_sdcp_gb300 import synth
    off = batch.m_offsets.detach().cpu().numpy().astype(np.int64)
    trows, drows, offs = [], [], [0]
    for b in sessions:
        o0, o1 = int(off[b]), int(off[b + 1])
        trows.extend(range(o0 + b, o1 + b + 1))
        drows.extend(range(o0, o1))
        offs.append(offs[-1] + (o1 - o0))
    dev = batch.target.device
    ti = torch.as_tensor(trows, dtype=torch.long, device=dev)
    di = torch.as_tensor(drows, dtype=torch.long, device=dev)
    T = synth.to_numpy_logits(batch.target.index_select(0, ti))
    D = synth.to_numpy_logits(batch.draft.index_select(0, di))
    x = batch.draft_tokens.index_select(0, di).cpu().numpy().astype(np.int32)
    return T, D, np.asarray(offs, np.int32), x, batch.params[list(sessions)]


def time_oracle(batch, seconds: float, cores: int, per_call: int):
    """Run the oracle over successive groups of `per_call` sessions until `seconds` pass."""
    import oracle
    oracle.build()
    B = batch.B
    groups, toks, elapsed, calls = [], 0, 0.0, 0
    start = 0
    while elapsed < seconds or calls == 0:
        sess = [(start + i) % B for i in range(min(per_call, B))]
        start = (start + per_call) % B
        args = oracle_sessions(batch, sess)
        t0 = time.perf_counter()
        r = oracle.verify_batch(*args, nthreads=cores, want_detail=False)
        elapsed += time.perf_counter() - t0
        toks += int(r["n_out"].sum())
        calls += 1
        groups.append(len(sess))
    return toks, elapsed, calls, sum(groups)


# ------------------------------------------------------------------------------------------
# the GPU arm
# ------------------------------------------------------------------------------------------
def run_ours(args, dist: Dist):
    import numpy as np
    import torch
    from speculative_decoding_verification_sdcp_gb300 import synth
    try:
        from speculative_decoding_verification_sdcp_gb300 import sdcp as binding
    except ImportError:
        from speculative_decoding_verification_sdcp_gb300 import build_ext
        build_ext.build()
        from speculative_decoding_verification_sdcp_gb300 import sdcp as binding
    assert torch.cuda.is_available(), "the GPU arm needs a CUDA device"
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    batch = synth.make_batch(w, device=dev, max_sessions=args.sessions)
    ver = binding.Verifier(batch.V, batch.B, batch.total_drafts, dev)
    ab = synth.algorithmic_bytes(batch)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ver(batch.target, batch.draft, batch.m_offsets, batch.draft_tokens, batch.params_dev)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    tokens_per_step = int(ver.n_out.sum().item())
    status_ok = int((ver.status == 0).sum().item())

    # ---- timed region: exactly K steps, events on the launching stream ---------------
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.05)
    dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()              # L2 flush between timed steps (outside the events)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_mean = sum(step_ms) / K
    ms_max_ranks = dist.reduce(ms_mean, "max")
    tokens_all = dist.reduce(float(tokens_per_step), "sum")
    value = tokens_all / (ms_max_ranks * 1e-3)
    launches = 2 * K

    # ---- kernel split (same two launches, an event between the phases) ---------------
    KS = min(K, 500)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(KS)]
    for i in range(KS):
        flush.zero_()
        evs[i][0].record(stream)
        ver.phases(batch.target, batch.draft, batch.m_offsets, batch.draft_tokens, batch.params_dev,
                   ev_mid=evs[i][1])
        evs[i][2].record(stream)
    torch.cuda.synchronize()
    rows_ms = sum(a.elapsed_time(b) for a, b, _ in evs) / KS
    sess_ms = sum(b.elapsed_time(c) for _, b, c in evs) / KS
    peak, peak_kind = measured_peaks()
    achieved = ab["bytes_rows"] / (rows_ms * 1e-3) / 1e9
    traffic = profiled_traffic(args.workload)

    # ---- end to end through the C ABI from pinned host buffers ----------------------------
    e2e = None
    if not args.no_e2e:
        h_t = batch.target.cpu().pin_memory()
        h_d = batch.draft.cpu().pin_memory()
        h_o = batch.m_offsets.cpu().pin_memory()
        h_x = batch.draft_tokens.cpu().pin_memory()
        h_p = batch.params_dev.cpu().pin_memory()
        d_t, d_d = torch.empty_like(batch.target), torch.empty_like(batch.draft)
        d_o, d_x, d_p = torch.empty_like(batch.m_offsets), torch.empty_like(batch.draft_tokens), torch.empty_like(batch.params_dev)
        o_acc = torch.empty(batch.B, dtype=torch.int32).pin_memory()
        o_n = torch.empty(batch.B, dtype=torch.int32).pin_memory()
        o_tok = torch.empty(batch.total_drafts + batch.B, dtype=torch.int32).pin_memory()
        o_st = torch.empty(batch.B, dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (h_t, h_d, h_o, h_x, h_p))
        d2h = sum(t.numel() * t.element_size() for t in (o_acc, o_n, o_tok, o_st))
        KE = max(3, min(K, 50))
        e_ms = []
        for i in range(KE + 2):
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for src, dst in ((h_t, d_t), (h_d, d_d), (h_o, d_o), (h_x, d_x), (h_p, d_p)):
                dst.copy_(src, non_blocking=True)
            ver(d_t, d_d, d_o, d_x, d_p)
            o_acc.copy_(ver.accepted, non_blocking=True)
            o_n.copy_(ver.n_out, non_blocking=True)
            o_tok.copy_(ver.out_tokens, non_blocking=True)
            o_st.copy_(ver.status, non_blocking=True)
            b_.record(stream)
            b_.synchronize()
            if i >= 2:
                e_ms.append(a.elapsed_time(b_))
        assert int(o_n.sum()) == tokens_per_step
        e_mean = sum(e_ms) / len(e_ms)
        e_max = dist.reduce(e_mean, "max")
        e2e = {"value": tokens_all / (e_max * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_max}

    # ---- CPU oracle on the host cores (rank 0, N = 1) --------------------------------------
    cpu = None
    if not args.no_cpu_baseline and dist.world == 1 and dist.rank == 0:
        cores = len(os.sched_getaffinity(0))
        toks, secs, calls, sess = time_oracle(batch, args.cpu_seconds, cores, per_call=min(batch.B, cores))
        cpu = {"value": toks / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "%d sessions of the same batch (%d oracle calls of %d sessions, %.1f s, fp64 C with OpenMP)" % (
                   sess, calls, min(batch.B, cores), secs)}

    if dist.rank == 0:
        M = np.diff(batch.m_offsets.cpu().numpy())
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_max_ranks, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name if args.sessions is None else "%s (first %d sessions)" % (w.name, batch.B),
                       "description": w.note, "B": batch.B, "V": batch.V,
                       "total_drafts": batch.total_drafts, "logits_dtype": "bf16" if batch.dtype_code == 1 else "f32",
                       "l2": "flushed between timed steps (256 MiB write)",
                       "parallelism": "sessions sharded by GPU (dp%d)" % dist.world},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "kernel": "row_stats_kernel",
                         "peak_kind": peak_kind + " copy bandwidth",
                         "algorithmic_bytes_per_launch": ab["bytes_rows"], "kernel_ms": rows_ms},
            "phases_ms": {"row_stats": rows_ms, "sessions": sess_ms},
            "step_gbps_algorithmic": (ab["bytes_rows"] + ab["bytes_extra_row_per_session"]) / (ms_max_ranks * 1e-3) / 1e9,
            "tokens_per_step": tokens_per_step, "sessions_ok": status_ok,
            "mean_tokens_per_session": tokens_per_step / batch.B,
            "m_histogram": {str(int(k)): int(v) for k, v in zip(*np.unique(M, return_counts=True))},
            "step_ms_median": statistics.median(step_ms), "wall_s_timed": wall,
            "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
            "gpu_launches": launches,
            "e2e": e2e, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# the reference arm: the CPU oracle, as it stands, on the host cores
# ------------------------------------------------------------------------------------------
def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return
    import torch
    from speculative_decoding_verification_sdcp_gb300 import synth
    import oracle
    oracle.build()
    w = synth.WORKLOADS[args.workload]
    dev = "cuda:%d" % dist.local if torch.cuda.is_available() else "cpu"
    batch = synth.make_batch(w, device=dev, max_sessions=args.sessions)
    cores = len(os.sched_getaffinity(0))
    per = min(batch.B, cores)
    B = batch.B
    samples = []
    cursor = 0
    for i in range(args.warmup + args.steps):
        sess = [(cursor + j) % B for j in range(per)]
        cursor = (cursor + per) % B
        samples.append(oracle_sessions(batch, sess))
        if len(samples) > 16:
            break
    tok, secs = 0, 0.0
    for i in range(args.warmup):
        oracle.verify_batch(*samples[i % len(samples)], nthreads=cores, want_detail=False)
    t_all = []
    for i in range(args.steps):
        s = samples[i % len(samples)]
        t0 = time.perf_counter()
        r = oracle.verify_batch(*s, nthreads=cores, want_detail=False)
        dt = time.perf_counter() - t0
        t_all.append(dt)
        tok += int(r["n_out"].sum())
        secs += dt
    value = tok / secs
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": w.name, "description": w.note,
                       "sample_per_step": "%d sessions of the batch" % per},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "%d sessions per step, %d steps" % (per, args.steps)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    dist = Dist(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
