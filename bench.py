#!/usr/bin/env python3
"""Benchmark of the batched acceptance step (libsdcp on GB300).

One step = one sdcp_verify_batch call over one synthetic verify batch (all phases:
row statistics of the sampling profile, acceptance tests, first-rejection scan, draw of
the additional token).  Default (headline) workload: the largest single-GPU batch,
B=32 sessions, M=64, V=262144, fp32 logits, speculative sampling over the full
distribution.  The line's per_config block times the three other large workloads
(topk50, topp90_ragged, large_batch_mixed) whole, under the same rules.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  value = verified tokens/s (sum of n_out over the batch,
summed over ranks, divided by the max over ranks of the mean device time of a step;
inputs resident in HBM; L2 flushed by a 256 MiB write between timed steps).
N > 1 runs under torchrun, one process per GPU: the batch is split into N contiguous
blocks of sessions balanced by scored rows (sdcp_split_sessions) and each GPU verifies
its block (strong scaling; sessions are independent, no collective on the data path).
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
DEFAULT_WORKLOAD = "mmax_stress"
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
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the headline workload (no per_config block)")
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
def load_binding():
    try:
        from speculative_decoding_verification_sdcp_gb300 import sdcp as binding
    except ImportError:
        from speculative_decoding_verification_sdcp_gb300 import build_ext
        build_ext.build()
        from speculative_decoding_verification_sdcp_gb300 import sdcp as binding
    return binding


def rank_batch(name, dist, dev, sessions=None):
    """The workload's batch on this rank: the whole batch at N = 1; under torchrun the
    rank's contiguous block of sessions (sdcp_split_sessions, balanced by scored rows)."""
    from speculative_decoding_verification_sdcp_gb300 import synth
    binding = load_binding()
    batch = synth.make_batch(synth.WORKLOADS[name], device=dev, max_sessions=sessions)
    bounds = None
    if dist.world > 1:
        bounds = binding.sdcp_split_sessions(batch.m_offsets.cpu().numpy(), batch.params, dist.world)
        lo, hi = int(bounds[dist.rank]), int(bounds[dist.rank + 1])
        batch = synth.shard_batch(batch, lo, hi)
    return batch, bounds


def measure(name, args, dist, dev, flush, K, sessions=None, want_e2e=False):
    """Device-timed steps of one workload (plus the phase split, a back-to-back call rate
    and, optionally, the end-to-end leg); returns the per-workload figures."""
    import numpy as np
    import torch
    from speculative_decoding_verification_sdcp_gb300 import synth
    binding = load_binding()
    batch, bounds = rank_batch(name, dist, dev, sessions)
    ver = binding.Verifier(batch.V, batch.B, batch.total_drafts, dev)
    ab = synth.algorithmic_bytes(batch)
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
    rows_bytes_all = dist.reduce(float(ab["bytes_rows"]), "sum")
    extra_bytes_all = dist.reduce(float(ab["bytes_extra_row_per_session"]), "sum")

    # ---- kernel split (same two launches, an event between the phases) ---------------
    KS = max(3, min(K, 500))
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

    # ---- back-to-back calls, no flush: host wall clock per call (launch cost included) --
    NB = max(10, min(200, K))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(NB):
        step()
    torch.cuda.synchronize()
    b2b_us = (time.perf_counter() - t0) / NB * 1e6

    step_gbps = (rows_bytes_all + extra_bytes_all) / (ms_max_ranks * 1e-3) / 1e9
    res = {
        "workload": name, "B": batch.B, "V": batch.V, "total_drafts": batch.total_drafts,
        "logits_dtype": "bf16" if batch.dtype_code == synth.BF16 else "f32",
        "value": tokens_all / (ms_max_ranks * 1e-3), "ms_per_step": ms_max_ranks,
        "step_ms_median": statistics.median(step_ms), "wall_s_timed": wall,
        "tokens_per_step": tokens_per_step, "tokens_all_ranks": tokens_all, "sessions_ok": status_ok,
        "rows_ms": rows_ms, "sessions_ms": sess_ms,
        "row_kernel_gbps": achieved, "row_kernel_frac": achieved / peak,
        "step_gbps_algorithmic": step_gbps, "step_frac": step_gbps / peak,
        "back_to_back_us_per_call": b2b_us,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "_peak": peak, "_peak_kind": peak_kind, "_ab": ab, "_K": K, "_batch": batch, "_ver": ver,
        "_bounds": None if bounds is None else [int(v) for v in bounds],
        "_M": np.diff(batch.m_offsets.cpu().numpy()),
    }
    if want_e2e:
        res["e2e"] = measure_e2e(batch, ver, stream, K, tokens_per_step, tokens_all, dist)
    return res


def measure_e2e(batch, ver, stream, K, tokens_per_step, tokens_all, dist):
    """The same metric through the public call with host buffers: every step copies its
    inputs from pinned host memory (one cudaMemcpyAsync per buffer) and reads its results
    back, inside the timed region."""
    import torch
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
    ins = ((h_t, d_t), (h_d, d_d), (h_o, d_o), (h_x, d_x), (h_p, d_p))
    h2d = sum(h.numel() * h.element_size() for h, _ in ins)
    d2h = sum(t.numel() * t.element_size() for t in (o_acc, o_n, o_tok, o_st))
    KE = max(3, min(K, 20))
    e_ms, c_ms = [], []
    for i in range(KE + 2):
        a, m, b_ = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        for src, dst in ins:
            dst.copy_(src, non_blocking=True)
        m.record(stream)
        ver(d_t, d_d, d_o, d_x, d_p)
        o_acc.copy_(ver.accepted, non_blocking=True)
        o_n.copy_(ver.n_out, non_blocking=True)
        o_tok.copy_(ver.out_tokens, non_blocking=True)
        o_st.copy_(ver.status, non_blocking=True)
        b_.record(stream)
        b_.synchronize()
        if i >= 2:
            e_ms.append(a.elapsed_time(b_))
            c_ms.append(a.elapsed_time(m))
    assert int(o_n.sum()) == tokens_per_step
    e_mean = sum(e_ms) / len(e_ms)
    e_max = dist.reduce(e_mean, "max")
    c_mean = sum(c_ms) / len(c_ms)
    return {"value": tokens_all / (e_max * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e_max, "h2d_ms": c_mean,
            "h2d_gbps": h2d / (c_mean * 1e-3) / 1e9, "steps": KE}


PER_CONFIG = ["topk50", "topp90_ragged", "large_batch_mixed", "mmax_stress"]


def run_ours(args, dist: Dist):
    import torch
    from speculative_decoding_verification_sdcp_gb300 import synth
    assert torch.cuda.is_available(), "the GPU arm needs a CUDA device"
    load_binding()
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    K = args.steps

    head = measure(args.workload, args, dist, dev, flush, K, sessions=args.sessions,
                   want_e2e=not args.no_e2e)
    batch, ab, peak = head["_batch"], head["_ab"], head["_peak"]
    traffic = profiled_traffic(args.workload) if args.sessions is None and dist.world == 1 else None

    # ---- CPU oracle on the host cores (rank 0, N = 1) --------------------------------------
    cpu = None
    if not args.no_cpu_baseline and dist.world == 1 and dist.rank == 0:
        cores = len(os.sched_getaffinity(0))
        toks, secs, calls, sess = time_oracle(batch, args.cpu_seconds, cores, per_call=min(batch.B, cores))
        cpu = {"value": toks / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "%d sessions of the same batch (%d oracle calls of %d sessions, %.1f s, fp64 C with OpenMP)" % (
                   sess, calls, min(batch.B, cores), secs)}
    head_launches = 2 * K  # the row kernel and the session kernel of every step
    del head["_batch"], head["_ver"]
    torch.cuda.empty_cache()

    # ---- the other target workloads, each whole, same timing rules ---------------------------
    per_config = {}
    if not args.no_per_config and args.sessions is None:
        for name in PER_CONFIG:
            if name == args.workload:
                continue
            r = measure(name, args, dist, dev, flush, K)
            for k in [k for k in r if k.startswith("_")]:
                del r[k]
            per_config[name] = r
            torch.cuda.empty_cache()

    if dist.rank == 0:
        import numpy as np
        w = synth.WORKLOADS[args.workload]
        M = head["_M"]
        parallelism = ("one GPU" if dist.world == 1 else
                       "sessions split into %d contiguous blocks balanced by scored rows, one per GPU, "
                       "no collective on the data path (bounds %s)" % (dist.world, head["_bounds"]))
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": dist.world, "steps": K,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name if args.sessions is None else "%s (first %d sessions)" % (w.name, batch.B),
                       "description": w.note, "B": w.B if args.sessions is None else batch.B, "V": batch.V,
                       "logits_dtype": head["logits_dtype"],
                       "arithmetic": "fp32 statistics and weights, fp64 acceptance compare",
                       "l2": "flushed between timed steps (256 MiB write)",
                       "parallelism": parallelism},
            "roofline": {"bound": "hbm", "achieved": head["row_kernel_gbps"], "peak": peak, "unit": "GB/s",
                         "frac": head["row_kernel_frac"], "traffic": traffic, "kernel": "row_stats_kernel",
                         "peak_kind": head["_peak_kind"] + " copy bandwidth (read+write copy; a read-only stream can exceed it)",
                         "algorithmic_bytes_per_launch": ab["bytes_rows"], "kernel_ms": head["rows_ms"]},
            "phases_ms": {"row_stats": head["rows_ms"], "sessions": head["sessions_ms"]},
            "step_gbps_algorithmic": head["step_gbps_algorithmic"], "step_frac": head["step_frac"],
            "tokens_per_step": head["tokens_all_ranks"], "sessions_ok": head["sessions_ok"],
            "mean_tokens_per_session": head["tokens_per_step"] / batch.B,
            "m_histogram": {str(int(k)): int(v) for k, v in zip(*np.unique(M, return_counts=True))},
            "step_ms_median": head["step_ms_median"], "wall_s_timed": head["wall_s_timed"],
            "back_to_back_us_per_call": head["back_to_back_us_per_call"],
            "clocks": head["clocks"],
            "gpu_launches": head_launches,
            "e2e": head.get("e2e"), "cpu_baseline": cpu,
            "per_config": per_config,
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
    # distinct groups of `per` sessions, at most four held on the host at once (a group of
    # the largest workload is about 2 GB); steps cycle over them
    samples = []
    cursor = 0
    for i in range(min(args.warmup + args.steps, (B + per - 1) // per, 4)):
        sess = [(cursor + j) % B for j in range(per)]
        cursor = (cursor + per) % B
        samples.append(oracle_sessions(batch, sess))
    del batch
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
            "scaling": "strong", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
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
