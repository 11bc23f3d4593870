"""Benchmark: one decode step (KV append + paged decode attention) on GB300.

Default workload: the Llama-3-8B-shaped GQA batch (B=64, 32 q / 8 kv heads,
D=128, bf16, 16-token blocks, lengths log-uniform in [512, 32768], pool 1.1x
the blocks in use), seeded synthetic data. One step = pa_append_kv of the new
token of every sequence + pa_decode over all tokens. The pools (~2 GB) are
larger than L2, so no flush is needed between steps.

Prints one JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle
on the host cores instead, on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak), queries·heads/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 2**20

# DRAM traffic of the split-attention kernel from an ncu capture (per launch,
# scaled to the full workload), valid only for the kernel sources it was
# measured on (sha256 of the split kernel's source files).
TRAFFIC = {"source_sha": "dada515cdcaf5f7fe87024fae57afc2148cf5706c625c1a023417ca97de38170",
           "workload": "llama3_8b_gqa", "bytes_per_launch": 2205629824 + 5011456}


def split_source_sha() -> str:
    h = hashlib.sha256()
    for name in ("pa_split.cuh", "pa_split.cu", "pa_ptx.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_202_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def CONFIGS_NEW_TOKENS(name):
    from paged_kv_cache_202_gb300.workloads import CONFIGS
    return CONFIGS[name].get("new_tokens", 256)


FALLBACK_BF16_TFLOPS = 1900.0
LATENCY_GRAPH_STEPS = 20  # steps per CUDA graph in the latency row


def measured_peak_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("bf16_tflops", "bf16_TFLOPs"):
            if key in d:
                v = d[key]
                if isinstance(v, dict):
                    v = v.get("burst", v.get("value"))
                return float(v), "measured"
    except (OSError, ValueError, TypeError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def measured_peak_tflops_sustained():
    """The bf16 GEMM rate held back to back for seconds (clocks under the power cap), or None."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = json.load(f).get("bf16_tflops_sustained")
        return float(v) if v is not None else None
    except (OSError, ValueError, TypeError):
        return None


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_gb_s"):
            if key in d:
                v = d[key]
                if isinstance(v, dict):
                    v = v.get("burst", v.get("value"))
                return float(v), "measured"
    except (OSError, ValueError, TypeError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples in the background (timestamps in ms)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:
            inside = [p for (_, p) in self.samples]
            window = "run"
        if not inside:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower() in ("active", "1")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window}


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def oracle_step_state(wl):
    """CPU-baseline leg: the workload after the step's append, as the oracle
    computes it (``oracle.append`` on copies of the host pools)."""
    import dataclasses
    import oracle
    oracle.build()
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.append(wl.k_new, wl.v_new, kp, vp, wl.block_tables, wl.cache_lens)
    return dataclasses.replace(wl, k_pool=kp, v_pool=vp)


def oracle_sample_gbs(wl, sample_s: float, min_pairs: int = 1):
    """Time the fp64 oracle on (b, h) pairs of the workload for about sample_s.

    ``wl`` holds the pools after the append (``oracle_step_state``). Returns
    (GB/s of algorithmic bytes, seconds, pairs, threads). The bytes of one
    (b, h) pair are sequence b's decode bytes divided by Hq.
    """
    import oracle
    import paged_kv_cache_202_gb300 as pa
    kp, vp = wl.k_pool, wl.v_pool
    threads = os.cpu_count() or 1
    eb = wl.elem_bytes
    per_seq = [pa.decode_bytes([int(L)], wl.Hq, wl.Hkv, wl.D, wl.block_size, eb, eb) / wl.Hq
               for L in wl.seq_lens]
    order = np.random.default_rng(0).permutation(wl.B * wl.Hq)
    # Random rows, cycling through the whole workload until the time is spent.
    pairs, done_bytes, elapsed, i = 0, 0.0, 0.0, 0
    chunk = max(min_pairs, threads)
    while elapsed < sample_s or pairs < min_pairs:
        if i >= order.size:
            i = 0
        sel = order[i:i + chunk]
        i += chunk
        pr = np.stack([sel // wl.Hq, sel % wl.Hq], axis=1).astype(np.int32)
        t = time.perf_counter()
        oracle.decode(wl.q, kp, vp, wl.block_tables, wl.seq_lens, wl.scale, pairs=pr,
                      nthreads=threads)
        elapsed += time.perf_counter() - t
        pairs += len(sel)
        done_bytes += sum(per_seq[int(b)] for b in sel // wl.Hq)
        chunk = min(chunk * 2, 4096)
    return done_bytes / elapsed / 1e9, elapsed, pairs, threads


def aggregate_over_ranks(world: int, seconds: float, units: float, device) -> tuple[float, float]:
    """Whole-job figures of `world` replica ranks (one process per GPU, no
    data exchange): the slowest rank's time and the sum of the units every
    rank processed. With one rank the inputs come back unchanged. Every rank
    must call it (it is a collective when world > 1)."""
    if world == 1:
        return seconds, units
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


LAYOUTS = {"paged": "each sequence's blocks shuffled over the pool",
           "contiguous": "each sequence's blocks consecutive in the pool (same bits, renumbered)"}


STEPS = {"separate": "pa_append_kv + pa_decode",
         "fused": "pa_append_decode (the append inside the decode's split kernel)"}


def decode_config(wl, world: int, layout: str = "paged", step: str = "separate") -> dict:
    """The ``config`` of a decode-step line, the same for both arms."""
    return {"workload": wl.name, "layout": LAYOUTS[layout],
            "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D,
            "block_size": wl.block_size, "num_blocks": wl.num_blocks,
            "tokens": int(wl.seq_lens.sum()), "kv_dtype": wl.dtype,
            "l2": f"inputs larger than L2 ({2 * wl.k_pool.nbytes / 2**30:.2f} GiB of pools vs "
                  f"{L2_BYTES / 2**20:.0f} MiB L2), no flush",
            "step": STEPS[step], "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from paged_kv_cache_202_gb300.workloads import contiguous_layout, make_workload
    wl = make_workload(args.workload)
    if getattr(args, "layout", "paged") == "contiguous":
        wl = contiguous_layout(wl)
    wl = oracle_step_state(wl)
    total = args.steps + args.warmup
    per_step = max(0.05, min(20.0, 120.0 / max(total, 1)))
    vals = []
    t_all = 0.0
    pairs_all = 0
    threads = 1
    for step in range(total):
        gbs, el, pairs, threads = oracle_sample_gbs(wl, per_step)
        if step >= args.warmup:
            vals.append(gbs)
            t_all += el
            pairs_all += pairs
    value = statistics.median(vals) if vals else 0.0
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t_all / max(len(vals), 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(wl, world, args.layout, args.step),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{pairs_all} random (sequence, q-head) rows over "
                                   f"{len(vals)} steps, ~{per_step:.2f} s each"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline_leg(wl, out, args, bf: bool):
    """The oracle on the host cores: timed on a bounded sample of the
    workload (the CPU baseline), and its values on 64 sampled rows compared
    with the timed GPU output."""
    ref_wl = oracle_step_state(wl)
    parity = None
    if not args.no_parity:
        import oracle
        rng = np.random.default_rng(1)
        idx = rng.choice(wl.B * wl.Hq, size=min(64, wl.B * wl.Hq), replace=False)
        pr = np.stack([idx // wl.Hq, idx % wl.Hq], axis=1).astype(np.int32)
        ref = oracle.decode(ref_wl.q, ref_wl.k_pool, ref_wl.v_pool, wl.block_tables, wl.seq_lens,
                            wl.scale, pairs=pr)
        got = out.float().cpu().numpy()[pr[:, 0], pr[:, 1]].astype(np.float64)
        parity = {"rows": int(len(pr)), "max_abs_err": float(np.abs(got - ref).max()),
                  "tol": 1.5e-2 if bf else 2e-3}
    gbs, el, pairs, threads = oracle_sample_gbs(ref_wl, args.cpu_seconds)
    cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"{pairs} (sequence, q-head) rows ({pairs / (wl.B * wl.Hq):.1f} passes "
                     f"over the workload in random order), {el:.1f} s; bytes per row = its "
                     f"sequence's decode bytes / Hq"}
    return cpu, parity


def configure_plan(plan, args):
    """Explicit plan choices from the command line (merge mode, dynamic tail)."""
    import paged_kv_cache_202_gb300 as pa
    if args.merge != "auto":
        plan.set_merge({"kernel": pa.PA_MERGE_KERNEL, "fused": pa.PA_MERGE_FUSED}[args.merge])
    if args.schedule:
        permille, pages = (int(x) for x in args.schedule.split(","))
        plan.set_schedule(permille, pages)


# Seconds the timed region spans at least (--span): the K-step loop is
# repeated until it does, so that the clock sampler (one sample per 100 ms)
# sees it.
TIMED_SPAN_S = 2.0


# The other configurations, measured by the default run as well: each is
# this script run in a child process with its own flags (so that a failure
# there cannot touch the headline line), summarised under "extras".
EXTRA_RUNS = [
    ["--workload", "llama7b_mha", "--steps", "100", "--warmup", "10"],
    ["--workload", "mixed_shared", "--steps", "100", "--warmup", "10"],
    ["--workload", "long_splitk", "--steps", "20", "--warmup", "3"],
    ["--workload", "llama3_405b_gqa", "--steps", "50", "--warmup", "5"],
    ["--row", "spec", "--steps", "50", "--warmup", "5"],
    ["--row", "prefill", "--steps", "40", "--warmup", "5"],
]
EXTRA_TIMEOUT_S = 300


def run_extras() -> list:
    out = []
    for extra in EXTRA_RUNS:
        cmd = [sys.executable, os.path.join(ROOT, "bench.py"), *extra, "--span", "0.5",
               "--cpu-seconds", "2", "--no-extras"]
        t0 = time.time()
        entry = {"args": " ".join(extra)}
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=EXTRA_TIMEOUT_S)
            lines = [x for x in r.stdout.strip().splitlines() if x.startswith("{")]
            if r.returncode != 0 or not lines:
                entry["error"] = (r.stderr.strip().splitlines() or ["exit %d" % r.returncode])[-1][:300]
            else:
                d = json.loads(lines[-1])
                roof = d.get("roofline") or {}
                entry.update({
                    "row": d.get("row", "decode"), "workload": d["config"].get("workload"),
                    "metric": d.get("metric"), "value": d.get("value"), "unit": d.get("unit"),
                    "ms_per_step": d.get("ms_per_step"),
                    "kernel_ms": roof.get("ms_per_launch"), "frac": roof.get("frac"),
                    "peak": roof.get("peak"), "e2e": (d.get("e2e") or {}).get("value"),
                    "parity": d.get("parity"), "device_error": d.get("device_error"),
                    "clocks": {k: (d.get("clocks") or {}).get(k) for k in ("sm_mhz", "reasons")},
                })
        except subprocess.TimeoutExpired:
            entry["error"] = f"timed out after {EXTRA_TIMEOUT_S} s"
        except Exception as e:  # a malformed line: recorded, never fatal to the headline
            entry["error"] = repr(e)[:300]
        entry["wall_s"] = round(time.time() - t0, 1)
        out.append(entry)
    return out


def run_ours(args, rank, world, local_rank):
    import __graft_entry__
    import paged_kv_cache_202_gb300 as pa
    from paged_kv_cache_202_gb300.workloads import contiguous_layout, make_workload

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    overrides = {"B": args.sequences} if args.sequences else {}
    wl = make_workload(args.workload, seed=args.seed + rank if args.seed is not None else None,
                       **overrides)
    if args.layout == "contiguous":
        wl = contiguous_layout(wl)
    bf = wl.dtype == "bf16"

    def to_dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if bf else np.float32))
        return (t.view(torch.bfloat16) if bf else t).to(dev)

    q, k_new, v_new = to_dev(wl.q), to_dev(wl.k_new), to_dev(wl.v_new)
    k_pool, v_pool = to_dev(wl.k_pool), to_dev(wl.v_pool)
    tables = torch.from_numpy(wl.block_tables).to(dev)
    seq_lens = torch.from_numpy(wl.seq_lens).to(dev)
    cache_lens = torch.from_numpy(wl.cache_lens).to(dev)
    torch.cuda.synchronize()
    out_dtype = torch.bfloat16 if bf else torch.float32
    out = torch.empty(wl.B, wl.Hq, wl.D, dtype=out_dtype, device=dev)
    plan = pa.Plan()
    stream = torch.cuda.current_stream()
    max_len = wl.max_seq_len

    def calls(kn, vn, qq, bt, sl, cl, s, ev=None):
        """One step's calls: the append then the decode, or the fused call;
        ev = three events around (append, decode) for the kernel pass."""
        if ev:
            ev[0].record(s)
        if args.step == "fused":
            if ev:
                ev[1].record(s)
            pa.pa_append_decode(qq, kn, vn, k_pool, v_pool, bt, sl, wl.scale, out, max_len, plan,
                                s)
        else:
            pa.pa_append_kv(kn, vn, k_pool, v_pool, bt, cl, s)
            if ev:
                ev[1].record(s)
            pa.pa_decode(qq, k_pool, v_pool, bt, sl, wl.scale, out, max_len, plan, s)
        if ev:
            ev[2].record(s)

    def step():
        calls(k_new, v_new, q, tables, seq_lens, cache_lens, stream)

    step()                        # creates the plan
    configure_plan(plan, args)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pa.pa_last_device_error(plan) == 0 and pa.pa_last_device_error(None) == 0

    eb = wl.elem_bytes
    dec_bytes = pa.decode_bytes(wl.seq_lens, wl.Hq, wl.Hkv, wl.D, wl.block_size, eb, eb)
    app_bytes = pa.append_bytes(wl.B, wl.Hkv, wl.D, eb)
    step_bytes = dec_bytes + app_bytes

    # Repeats of the K-step loop: enough to span TIMED_SPAN_S, from a probe of
    # one K-step loop (the same on every rank: the slowest rank's probe).
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_a.record(stream)
    for _ in range(args.steps):
        step()
    e_b.record(stream)
    torch.cuda.synchronize()
    probe_ms, _ = aggregate_over_ranks(world, e_a.elapsed_time(e_b), 0, dev)
    repeats = max(1, min(100000, math.ceil(args.span * 1e3 / max(probe_ms, 1e-3))))

    # Timed region: R repeats of exactly K steps, each bracketed by a barrier
    # and a synchronize, issued exactly as a caller issues them. The split
    # and merge kernels start under programmatic dependent launch, which
    # overlaps each launch with its predecessor's drain; an event recorded
    # between two kernels would cancel that overlap, so the step loop carries
    # none.
    rep_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(repeats)]
    for a_, b_ in rep_ev:         # create the underlying events before the timed region
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    w0 = time.time()
    for a_, b_ in rep_ev:
        barrier()
        torch.cuda.synchronize()
        a_.record(stream)
        for _ in range(args.steps):
            step()
        b_.record(stream)
        torch.cuda.synchronize()
    w1 = time.time()
    barrier()
    # Kernel pass: the same number of steps again, with events around every
    # split launch, for the split kernel's average duration (the roofline
    # figure), and around the append and the whole decode call.
    k_steps = max(args.steps, min(repeats * args.steps, 3000))
    ev_split = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(k_steps)]
    ev_parts = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(k_steps)]
    for i in range(k_steps):
        for e in (*ev_split[i], *ev_parts[i]):
            e.record(stream)
    torch.cuda.synchronize()
    w2 = time.time()
    for i in range(k_steps):
        plan.set_split_events(*ev_split[i])
        calls(k_new, v_new, q, tables, seq_lens, cache_lens, stream, ev=ev_parts[i])
    torch.cuda.synchronize()
    w3 = time.time()
    plan.set_split_events(None, None)
    time.sleep(0.25)
    sampler.stop()
    # Per repeat: the slowest rank's time for K steps; every rank's bytes and query rows.
    rep_ms = []
    for a_, b_ in rep_ev:
        t, _ = aggregate_over_ranks(world, a_.elapsed_time(b_), 0, dev)
        rep_ms.append(t / args.steps)
    _, job_bytes = aggregate_over_ranks(world, 0.0, step_bytes, dev)
    _, job_qheads = aggregate_over_ranks(world, 0.0, wl.B * wl.Hq, dev)
    ms_step = statistics.median(rep_ms)
    split_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in ev_split)
    append_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev_parts)
    decode_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev_parts)
    err = pa.pa_last_device_error(plan)

    # End to end through the public API: inputs from pinned host memory each step,
    # result read back each step. The step's inputs (q, k_new, v_new, tables,
    # lengths) sit in one pinned staging buffer and cross in one copy, into
    # device views of one buffer that the calls read.
    parts = [q, k_new, v_new, tables, seq_lens, cache_lens]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(parts, offs):
        nb = t.numel() * t.element_size()
        h_in[o:o + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
        views.append(d_in[o:o + nb].view(t.dtype).view(t.shape))
    e_q, e_kn, e_vn, e_bt, e_sl, e_cl = views
    h_out = torch.empty_like(out, device="cpu").pin_memory()
    h2d = total
    d2h = h_out.numel() * h_out.element_size()
    e2e_steps = max(args.steps, min(2000, math.ceil(args.span * 1e3 / max(ms_step, 1e-3))))

    def e2e_calls(s):
        d_in.copy_(h_in, non_blocking=True)
        calls(e_kn, e_vn, e_q, e_bt, e_sl, e_cl, s)
        h_out.copy_(out, non_blocking=True)

    # The step's calls, warmed up once, then captured in a CUDA graph: every
    # e2e step replays the input copy, both calls and the result copy, and
    # waits for the result.
    e2e_calls(stream)
    torch.cuda.synchronize()
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph):
        e2e_calls(torch.cuda.current_stream())

    def e2e_step():
        e2e_graph.replay()
        torch.cuda.current_stream().synchronize()

    for _ in range(3):
        e2e_step()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s, _ = aggregate_over_ranks(world, (time.perf_counter() - t0) / e2e_steps, 0, dev)
    barrier()

    cpu, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, parity = cpu_baseline_leg(wl, out, args, bf)

    peak, peak_kind = measured_peak_gbs()
    achieved = dec_bytes / (split_ms * 1e-3) / 1e9
    sha = split_source_sha()
    # The recorded counters are the plain split kernel's: none for the fused
    # append's kernel or another layout.
    traffic = TRAFFIC["bytes_per_launch"] if TRAFFIC["source_sha"] == sha and \
        TRAFFIC["workload"] == wl.name and args.step == "separate" and \
        args.layout == "paged" else None
    value = job_bytes / (ms_step * 1e-3) / 1e9
    clocks = sampler.summary(w0, w1)
    clocks_kernel_pass = sampler.summary(w2, w3)
    path, blocks, warps = plan.info()
    plan.free()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "ms_per_step_min": min(rep_ms), "ms_per_step_max": max(rep_ms),
            "repeats": repeats,
            "timing": f"median over {repeats} repeats of the K-step loop (each bracketed by a "
                      f"barrier and a synchronize, timed by CUDA events on the launching "
                      f"stream), {1e-3 * sum(rep_ms) * args.steps:.2f} s timed in all",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
            if bf else "f32", "data": "synthetic",
            "config": decode_config(wl, world, args.layout, args.step),
            "pct_of_peak": 100.0 * value / world / peak,
            "qheads_per_s": job_qheads / (ms_step * 1e-3),
            "parts_ms": {"append": append_ms if args.step != "fused" else None,
                         "decode": decode_ms, "split_kernel": split_ms,
                         "timing": "CUDA events around each call in the kernel pass (events "
                                   "between calls, so no launch overlap); rank 0"},
            "roofline": {"bound": "hbm", "kernel": "split attention", "achieved": achieved,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "algorithmic_bytes": dec_bytes, "ms_per_launch": split_ms,
                         "timing": f"CUDA events around each of {k_steps} split launches, in "
                                   f"a second pass of as many steps"},
            "e2e": {"value": job_bytes / e2e_s / 1e9, "unit": "GB/s",
                    "ms_per_step": e2e_s * 1e3, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "how": "per step: the inputs from pinned host memory (one staging copy), "
                           "pa_append_kv, pa_decode, the output back, captured once in a CUDA "
                           "graph and replayed, then a wait for the result"},
            "gpu_launches": (2 if args.merge == "fused" or args.step == "fused" else 3)
            * args.steps * repeats,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "clocks_kernel_pass": clocks_kernel_pass,
            "parity": parity,
            "device_error": err,
            "kernel": {"path": {1: "simple", 2: "fma", 3: "mma"}.get(path, path),
                       "blocks": blocks, "warps": warps, "merge": args.merge,
                       "schedule": args.schedule or "auto"},
        }
        if world == 1 and not args.no_extras and args.layout == "paged" and args.step == "separate" \
                and args.workload == "llama3_8b_gqa" and args.merge == "auto" and args.schedule is None \
                and args.sequences is None:
            line["extras"] = run_extras()
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def row_cpu_baseline_leg(args, wl, out, qh, qs, ns):
    """CPU-baseline leg of the multi-query rows: the oracle's state after the
    step's append, its values on 24 sampled query rows compared with the
    GPU output, and the oracle timed on a bounded sample of the workload."""
    import oracle
    ref_wl = oracle_step_state(wl)
    parity = None
    if not args.no_parity:
        rng = np.random.default_rng(3)
        T = int(qs[-1])
        rows = rng.choice(T, size=min(24, T), replace=False)
        seq_of = np.searchsorted(qs, rows, side="right") - 1
        err = 0.0
        for r, b in zip(rows, seq_of):
            i = r - qs[b]
            sub = oracle.prefill(qh[r:r + 1], ref_wl.k_pool, ref_wl.v_pool,
                                 wl.block_tables[b:b + 1], [int(wl.seq_lens[b] - ns[b] + i + 1)],
                                 [0, 1], wl.scale)
            got = out[r].float().cpu().numpy().astype(np.float64)
            err = max(err, float(np.abs(got - sub[0]).max()))
        parity = {"rows": int(len(rows)), "max_abs_err": err, "tol": 1.5e-2}
    cpu = row_cpu_baseline(args.row, ref_wl, args.cpu_seconds, prefill_q=qh, prefill_qs=qs,
                           prefill_ns=ns)
    return cpu, parity


def row_cpu_baseline(row, wl, sample_s, prefill_q=None, prefill_qs=None, prefill_ns=None):
    """The oracle, as it stands, on a bounded random sample of the row's
    workload on the host cores (about sample_s of CPU work). For the
    multi-query rows ``wl`` holds the pools after the step's append."""
    import oracle
    rng = np.random.default_rng(5)
    elapsed, units, n = 0.0, 0.0, 0
    if row in ("prefill", "spec"):
        threads = os.cpu_count() or 1
        T = int(prefill_qs[-1])
        for r in np.tile(rng.permutation(T), max(1, 100000 // max(T, 1))):  # cycles until the time is spent
            b = int(np.searchsorted(prefill_qs, r, side="right") - 1)
            npos = int(wl.seq_lens[b] - prefill_ns[b] + (r - prefill_qs[b]) + 1)
            t = time.perf_counter()
            oracle.prefill(prefill_q[r:r + 1], wl.k_pool, wl.v_pool, wl.block_tables[b:b + 1],
                           [npos], [0, 1], wl.scale, nthreads=threads)
            elapsed += time.perf_counter() - t
            if row == "prefill":
                units += 4 * wl.D * wl.Hq * npos
            else:  # bytes: the sequence's K and V once, shared by its query rows
                units += 2 * wl.Hkv * wl.D * wl.elem_bytes * int(wl.seq_lens[b]) / prefill_ns[b]
            n += 1
            if elapsed >= sample_s:
                break
        scale, unit = (1e12, "TFLOP/s") if row == "prefill" else (1e9, "GB/s")
        return {"value": units / elapsed / scale, "unit": unit, "cores": threads,
                "kind": "oracle", "sample": f"{n} query rows (all {wl.Hq} heads each, random "
                                            f"order), {elapsed:.1f} s"}
    eb = wl.elem_bytes
    if row == "copy_blocks":
        block_bytes = wl.Hkv * wl.block_size * wl.D * eb
        perm = rng.permutation(wl.num_blocks).astype(np.int32)
        half = wl.num_blocks // 2
        batch = 0
        while elapsed < sample_s:
            k = batch % max(1, half // 64)
            batch += 1
            src, dst = perm[64 * k:64 * k + 64], perm[half + 64 * k:half + 64 * k + 64]
            t = time.perf_counter()
            oracle.copy_blocks(wl.k_pool, wl.v_pool, src, dst)
            elapsed += time.perf_counter() - t
            units += 2 * len(src) * block_bytes * 2
            n += len(src)
        what = f"{n} random block pairs in batches of 64"
    else:
        for b in np.tile(rng.permutation(wl.B), 1000):
            L = int(wl.seq_lens[b])
            t = time.perf_counter()
            oracle.page_scores(wl.k_pool, wl.v_pool, wl.block_tables[b:b + 1], wl.seq_lens[b:b + 1])
            elapsed += time.perf_counter() - t
            units += 2 * wl.Hkv * wl.D * eb * L
            n += 1
            if elapsed >= sample_s:
                break
        what = f"{n} sequences one at a time, random order"
    return {"value": units / elapsed / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{what}, {elapsed:.1f} s"}


def run_row(args, local_rank):
    """Measure one of the other hot-path kernels on the workload: whole-pool
    block copies (copy on write) or PagedEviction page scores."""
    import __graft_entry__
    import paged_kv_cache_202_gb300 as pa
    from paged_kv_cache_202_gb300.workloads import make_workload

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    overrides = {"B": args.sequences} if args.sequences else {}
    if args.seq_len:
        overrides.update(lengths=("fixed", args.seq_len), max_len=args.seq_len,
                         pool=("factor", 1.0))
    wl = make_workload(args.workload, **overrides)
    bf = wl.dtype == "bf16"

    def to_dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if bf else np.float32))
        return (t.view(torch.bfloat16) if bf else t).to(dev)

    k_pool, v_pool = to_dev(wl.k_pool), to_dev(wl.v_pool)
    tables = torch.from_numpy(wl.block_tables).to(dev)
    seq_lens = torch.from_numpy(wl.seq_lens).to(dev)
    eb = wl.elem_bytes
    if args.row != "copy_blocks":
        # The step's token goes into the device pools through the library's
        # append: every token a query or a page score reads is then cached.
        pa.pa_append_kv(to_dev(wl.k_new), to_dev(wl.v_new), k_pool, v_pool, tables,
                        torch.from_numpy(wl.cache_lens).to(dev))
        torch.cuda.synchronize()
    if args.row in ("prefill", "spec"):
        n_new = int(args.new_tokens or CONFIGS_NEW_TOKENS(args.workload))
        ns = np.minimum(wl.seq_lens, n_new).astype(np.int64)
        qs = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
        T = int(qs[-1])
        from paged_kv_cache_202_gb300.workloads import bf16_bits
        qh = bf16_bits(np.random.default_rng(7).standard_normal((T, wl.Hq, wl.D))
                       .astype(np.float32))
        q = to_dev(qh)
        q_start = torch.from_numpy(qs).to(dev)
        out = torch.empty(T, wl.Hq, wl.D, dtype=torch.bfloat16, device=dev)
        # causal: row i of sequence b sees L_b - n_b + i + 1 tokens; 4 D flops per token
        toks = sum(int(((wl.seq_lens[b] - ns[b] + 1) * 2 + ns[b] - 1) * ns[b] // 2)
                   for b in range(wl.B))
        flops = 4 * wl.D * wl.Hq * toks
        nbytes = 2 * wl.Hkv * wl.D * eb * int(wl.seq_lens.sum()) + 2 * T * wl.Hq * wl.D * 2

        if args.row == "prefill":
            def call():
                pa.pa_prefill(q, q_start, k_pool, v_pool, tables, seq_lens, wl.scale, out,
                              int(ns.max()), wl.max_seq_len)
        else:
            plan = pa.Plan()

            def call():
                pa.pa_decode_multi(q, q_start, k_pool, v_pool, tables, seq_lens, wl.scale, out,
                                   int(ns.max()), wl.max_seq_len, plan)
            call()                       # creates the plan
            configure_plan(plan, args)   # --schedule / --merge, for same-box comparisons
        what = f"{T} query rows ({n_new} newest tokens per sequence), causal"
    elif args.row == "copy_blocks":
        n = min(8192, wl.num_blocks // 2)
        perm = np.random.default_rng(0).permutation(wl.num_blocks)
        src = torch.from_numpy(perm[:n].astype(np.int32)).to(dev)
        dst = torch.from_numpy(perm[n:2 * n].astype(np.int32)).to(dev)
        block_bytes = wl.Hkv * wl.block_size * wl.D * eb
        nbytes = 2 * n * block_bytes * 2 + 8 * n  # both pools, read + write; the id lists

        def call():
            pa.pa_copy_blocks(k_pool, v_pool, src, dst)
        what = f"{n} random block pairs of {block_bytes} bytes per pool"
    else:
        B, MB = wl.block_tables.shape
        scores = torch.empty(B, MB, dtype=torch.float32, device=dev)
        victims = torch.empty(B, dtype=torch.int32, device=dev)
        nblk = sum(-(-int(L) // wl.block_size) for L in wl.seq_lens)
        nbytes = 2 * wl.Hkv * wl.D * eb * int(wl.seq_lens.sum()) + 4 * nblk + 4 * B + \
            4 * nblk + 4 * B  # K and V once, table entries, lengths, scores, victims

        def call():
            pa.pa_page_scores(k_pool, v_pool, tables, seq_lens, wl.max_seq_len, scores, victims)
        what = "every attended page of every sequence"
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for a_, b_ in ev:
        a_.record(stream)
        call()
        b_.record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in ev)
    peak, peak_kind = measured_peak_gbs()
    gbs = nbytes / (ms * 1e-3) / 1e9
    ms_graph = None
    if args.row in ("prefill", "spec"):
        # The same calls replayed from a CUDA graph: the device's own time per
        # call, without the host's per-call cost (which the events above
        # include when a call is shorter than its launch from Python).
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                for _ in range(LATENCY_GRAPH_STEPS):
                    call()
            reps = max(1, args.steps // LATENCY_GRAPH_STEPS)
            for _ in range(2):
                graph.replay()
            side.synchronize()
            t0.record(side)
            for _ in range(reps):
                graph.replay()
            t1.record(side)
            side.synchronize()
            ms_graph = t0.elapsed_time(t1) / (reps * LATENCY_GRAPH_STEPS)
            del graph
    if args.row in ("prefill", "spec"):
        tpeak, tkind = measured_peak_tflops()
        tfs = flops / (ms * 1e-3) / 1e12
        # Bound by arithmetic intensity: few queries per sequence (speculative
        # verification) make the pass HBM-bound, many (chunked prefill) tensor-bound.
        hbm_bound = flops / nbytes < tpeak * 1e12 / (peak * 1e9)
        cpu, parity = None, None
        if not args.no_cpu_baseline:
            cpu, parity = row_cpu_baseline_leg(args, wl, out, qh, qs, ns)
        print(json.dumps({
            "row": args.row,
            **({"metric": "prefill: achieved bf16 TFLOP/s", "value": tfs, "unit": "TFLOP/s"}
               if args.row == "prefill" else
               {"metric": "speculative verification (pa_decode_multi): achieved HBM GB/s",
                "value": gbs, "unit": "GB/s"}), "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "ms_per_step_graph": ms_graph,
            "value_graph": (flops / (ms_graph * 1e-3) / 1e12 if args.row == "prefill" else
                            nbytes / (ms_graph * 1e-3) / 1e9),
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "what": what, "queries_per_sequence": n_new,
                       "B": wl.B, "seq_len": args.seq_len or "the workload's"},
            "roofline": ({"bound": "hbm", "achieved": gbs, "peak": peak, "peak_kind": peak_kind,
                          "unit": "GB/s", "frac": gbs / peak, "algorithmic_bytes": nbytes,
                          "tflops": tfs} if hbm_bound else
                         {"bound": "tensor", "achieved": tfs, "peak": tpeak, "peak_kind": tkind,
                          "unit": "TFLOP/s", "frac": tfs / tpeak, "algorithmic_flops": flops,
                          "hbm_gbs": gbs,
                          # the same rate against the GEMM held for seconds, the fairer
                          # denominator when this loop runs long enough to meet the power cap
                          "peak_sustained": measured_peak_tflops_sustained(),
                          "frac_sustained": (tfs / measured_peak_tflops_sustained()
                                             if measured_peak_tflops_sustained() else None),
                          "timed_s": ms * args.steps * 1e-3}),
            "parity": parity,
            "gpu_launches": (2 if args.row == "spec" else 1) * (
                args.steps + args.warmup + LATENCY_GRAPH_STEPS * (2 + max(1, args.steps // LATENCY_GRAPH_STEPS))),
            "cpu_baseline": cpu,
        }), flush=True)
        return
    cpu = None if args.no_cpu_baseline else row_cpu_baseline(
        args.row, wl if args.row == "copy_blocks" else oracle_step_state(wl), args.cpu_seconds)
    print(json.dumps({
        "row": args.row, "metric": f"{args.row}: achieved HBM GB/s", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "what": what,
                   "l2": "inputs larger than L2, no flush"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": gbs / peak, "algorithmic_bytes": nbytes},
        "gpu_launches": (1 if args.row == "copy_blocks" else 2) * args.steps,
        "cpu_baseline": cpu,
    }), flush=True)


def run_latency(args, local_rank) -> None:
    """Step latency against sequence length at a fixed batch (context row).

    One append + decode step of the workload's head shape, every sequence of
    the same length, for lengths 128 .. 32768: where the step is bound by
    launch and latency and where by bandwidth. Plain calls on one stream,
    CUDA events around `steps` steps after `warmup`.
    """
    import __graft_entry__
    import paged_kv_cache_202_gb300 as pa
    from paged_kv_cache_202_gb300.workloads import make_workload
    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    B = args.batch
    lengths = [128 << k for k in range(9)]
    rows = []
    for L in lengths:
        wl = make_workload(args.workload, B=B, lengths=("fixed", L), max_len=L,
                           pool=("factor", 1.0))

        def to_dev(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        q, kn, vn = to_dev(wl.q), to_dev(wl.k_new), to_dev(wl.v_new)
        kp, vp = to_dev(wl.k_pool), to_dev(wl.v_pool)
        bt = torch.from_numpy(wl.block_tables).to(dev)
        sl = torch.from_numpy(wl.seq_lens).to(dev)
        cl = torch.from_numpy(wl.cache_lens).to(dev)
        out = torch.empty(wl.B, wl.Hq, wl.D, dtype=torch.bfloat16, device=dev)
        torch.cuda.synchronize()
        stream = torch.cuda.Stream(device=dev)  # graphs are captured on a stream of their own
        with torch.cuda.stream(stream), pa.Plan() as plan:
            def step():
                if args.step == "fused":
                    pa.pa_append_decode(q, kn, vn, kp, vp, bt, sl, wl.scale, out, L, plan, stream)
                else:
                    pa.pa_append_kv(kn, vn, kp, vp, bt, cl, stream)
                    pa.pa_decode(q, kp, vp, bt, sl, wl.scale, out, L, plan, stream)
            for _ in range(args.warmup):
                step()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                step()
            e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / args.steps
            # The same steps replayed from a CUDA graph: the device's own step
            # time, without the host's per-call cost (which bounds a loop of
            # eager calls from Python at short lengths).
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(LATENCY_GRAPH_STEPS):
                    step()
            reps = max(1, args.steps // LATENCY_GRAPH_STEPS)
            for _ in range(3):
                graph.replay()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            us_graph = e0.elapsed_time(e1) * 1e3 / (reps * LATENCY_GRAPH_STEPS)
            del graph
            assert pa.pa_last_device_error(plan) == 0
        eb = wl.elem_bytes
        nbytes = pa.decode_bytes(wl.seq_lens, wl.Hq, wl.Hkv, wl.D, wl.block_size, eb, eb) + \
            pa.append_bytes(wl.B, wl.Hkv, wl.D, eb)
        rows.append({"seq_len": L, "us_per_step": round(us, 2), "us_per_step_graph": round(us_graph, 2),
                     "gbs": round(nbytes / us / 1e3, 1), "gbs_graph": round(nbytes / us_graph / 1e3, 1)})
        del kp, vp
        torch.cuda.empty_cache()
    by = {r["seq_len"]: r["us_per_step"] for r in rows}
    print(json.dumps({
        "row": "latency", "metric": "decode step latency vs sequence length", "unit": "us",
        "value": by[2048], "higher_is_better": False, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D,
                   "block_size": wl.block_size, "step": STEPS[args.step]},
        "steps": args.steps, "warmup": args.warmup, "lengths": rows,
        "growth_128_to_2048": round(by[2048] / by[128], 3),
        "value_graph": {r["seq_len"]: r["us_per_step_graph"] for r in rows}[2048],
        "gpu_launches": (2 if args.step == "fused" else 3) * len(lengths) * (
            args.steps + args.warmup + (3 + max(1, args.steps // LATENCY_GRAPH_STEPS)) * LATENCY_GRAPH_STEPS),
        "timing": "CUDA events around `steps` back-to-back eager steps per length (us_per_step), "
                  "and around replays of a CUDA graph of %d steps (us_per_step_graph)" % LATENCY_GRAPH_STEPS,
    }))


def run_read_ceiling(args) -> None:
    """Read-only HBM ceiling beside the copy peak (`bench_read_ceiling.cu`).

    The decode step only reads its pools; the copy peak moves half its bytes
    as writes. A standalone CUDA program times a device-to-device copy, a
    streaming 16-byte read and a read of 4 KB pages in random order over the
    decode's 2.2 GB, and this leg prints its figures as one JSON line.
    """
    import paged_kv_cache_202_gb300 as pa
    from paged_kv_cache_202_gb300 import _build
    src = os.path.join(ROOT, "bench_read_ceiling.cu")
    exe = os.path.join(ROOT, "_build", "read_ceiling")
    if not os.path.exists(exe) or os.path.getmtime(exe) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(exe), exist_ok=True)
        r = subprocess.run([_build._nvcc(), *_build.ARCH, "-O3", "-std=c++17", src, "-o", exe],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for bench_read_ceiling.cu:\n{r.stderr}")
    from paged_kv_cache_202_gb300.workloads import CONFIGS, workload_lengths
    cfg = CONFIGS[args.workload]
    eb = 2 if cfg["dtype"] == "bf16" else 4
    dec_bytes = pa.decode_bytes(workload_lengths(args.workload, args.seed), cfg["Hq"], cfg["Hkv"],
                                cfg["D"], cfg["block_size"], eb, eb)
    pages = -(-dec_bytes // 4096)
    r = subprocess.run([exe, str(pages), str(max(args.steps, 3))], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"read_ceiling exited {r.returncode}: {r.stderr.strip()}")
    d = json.loads(r.stdout.strip().splitlines()[-1])
    res = {x["name"]: x for x in d["results"]}
    stream = max((x for x in d["results"] if x["name"].startswith("stream_")),
                 key=lambda x: x["median_gbs"])
    pages = max((x for x in d["results"] if x["name"].startswith("pages_")),
                key=lambda x: x["median_gbs"])
    peak, kind = measured_peak_gbs()
    print(json.dumps({
        "row": "read_ceiling", "metric": "read-only HBM GB/s (streaming, 16-byte loads)",
        "value": stream["median_gbs"], "unit": "GB/s", "n_gpus": 1, "steps": d["reps"],
        "higher_is_better": True, "dtype": "u8", "data": "synthetic",
        "config": {"workload": "read_ceiling", "bytes": d["bytes"],
                   "sized_as": f"one decode of {args.workload} ({dec_bytes} bytes), in 4 KB pages",
                   "l2": f"buffer {d['bytes'] / L2_BYTES:.1f}x the L2, no flush"},
        "pages_4k_random_gbs": pages["median_gbs"], "copy_d2d_gbs": res["copy_d2d"]["median_gbs"],
        "copy_peak": {"value": peak, "kind": kind},
        "stream_over_copy_peak": stream["median_gbs"] / peak,
        "pages_over_copy_peak": pages["median_gbs"] / peak,
        "results": d["results"], "gpu_launches": (len(d["results"]) - 1) * (d["reps"] + 3),
        "timing": "each launch timed alone by CUDA events; median of `steps` launches after 3 warm-up",
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None,
                    help="default: llama3_8b_gqa (prefill row: prefill_gqa)")
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other configurations the default run also measures")
    ap.add_argument("--span", type=float, default=TIMED_SPAN_S,
                    help="seconds the timed region spans at least (0: exactly K steps, "
                         "e.g. under a profiler)")
    ap.add_argument("--merge", default="auto", choices=["auto", "kernel", "fused"],
                    help="how the decode combines split partials (pa_plan_set_merge)")
    ap.add_argument("--schedule", default=None,
                    help="permille,pages: force the dynamic tail (pa_plan_set_schedule)")
    ap.add_argument("--new-tokens", type=int, default=None,
                    help="prefill / spec rows: queries per sequence (default: the workload's)")
    ap.add_argument("--step", default="separate", choices=sorted(STEPS),
                    help="decode row: the step's calls (fused = pa_append_decode)")
    ap.add_argument("--layout", default="paged", choices=sorted(LAYOUTS),
                    help="decode row: the pool layout (contiguous = every sequence's blocks "
                         "consecutive, the unpaged baseline of the paging cost)")
    ap.add_argument("--row", default="decode",
                    choices=["decode", "copy_blocks", "page_scores", "prefill", "spec",
                             "read_ceiling", "latency"])
    ap.add_argument("--batch", type=int, default=1,
                    help="latency row: sequences per step (all of one length)")
    ap.add_argument("--sequences", type=int, default=None,
                    help="decode and other rows: N sequences drawn by the workload's recipe (a "
                         "smaller case of the same workload, e.g. for a profiler capture or a "
                         "small batch)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="rows other than decode: every sequence of this many tokens")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload is None:
        args.workload = {"prefill": "prefill_gqa", "spec": "spec_gqa",
                         "latency": "llama7b_mha"}.get(args.row, "llama3_8b_gqa")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.row == "read_ceiling":
        run_read_ceiling(args)
    elif args.row == "latency":
        run_latency(args, local_rank)
    elif args.row != "decode":
        run_row(args, local_rank)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
