"""Benchmark: paged decode effective KV HBM GB/s (and % of peak), prefill TFLOP/s.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line.  The headline `value` is the effective KV bandwidth of
paged_decode_run on the Llama-3-8B-shaped decode workload (B=64, Hq=32,
Hkv=8, D=128, page_size=16, kv_len U[512, 8192], 40K-page shuffled pool):
algorithmic K+V bytes of the visited tokens / device time per call, with the
inputs resident in HBM (each call reads ~1.1 GB, far more than the 129 MB L2,
so no flush is needed).  The other decode workloads and the ragged prefill are
measured in the same run and reported as sub-objects.

Under torchrun (N > 1) every rank decodes its own batch of the same shape
(weak scaling, no collective on the data path); `value` sums the bytes of all
ranks over the slowest rank's time.
"""

import argparse
import datetime
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "llama3_8b"
PREFILL_WINDOW = 2047   # sliding-window variant of the ragged prefill (2048 keys per row)
# DRAM read + write bytes of one headline decode launch (decode_mma_kernel<2>
# with the transposed step of groups of at most 8 rows, seed 0, one GB300):
# ncu's dram__bytes_read.sum + dram__bytes_write.sum for that launch, captured
# on this same command (one metric pass, full size).  Other seeds or ranks
# scale it by their algorithmic K+V bytes.
# the kernel symbol each decode plan launches
KERNEL_SYMBOL = {"cuda_core": "decode_cc_kernel", "mma": "decode_mma_kernel"}
NCU_TRAFFIC = {"kernel": "decode_mma_kernel", "kv_bytes": 1128361984,
               "dram_bytes": 1130968064 + 4109824}
METRIC = "paged decode effective KV HBM GB/s"
UNIT = "GB/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--workload", default=None,
                    help="profiling: time only this decode workload (llama3_8b, skewed, spec), "
                         "'prefill', 'prefill_variable_window' or 'merge'")
    ap.add_argument("--batch", type=int, default=None,
                    help="profiling: override the workload's batch size (smaller capture; "
                         "for 'merge', the rows per state)")
    ap.add_argument("--mma-min-rows", type=int, default=0,
                    help="decode plan: rows per KV head from which the mma kernel is used")
    ap.add_argument("--split-waves", type=int, default=0,
                    help="decode plan: target CTAs = split_waves x SMs (0 = library default)")
    ap.add_argument("--dtype", choices=["bf16", "f16"], default="bf16",
                    help="profiling: q/K/V type of the one decode workload timed")
    ap.add_argument("--head-dim", type=int, default=128, choices=[128, 256],
                    help="profiling: head_dim of the 'prefill' workload")
    ap.add_argument("--seed", type=int, default=0)
    return ap.parse_args()


PLAN_OVERRIDES = {}


def profile_case(args):
    """One workload only (for ncu captures and sweeps); prints a short JSON line."""
    import torch
    from paged_kv_attention_32_gb300 import workloads as wl
    peak_gbs, peak_tf, _ = measured_peaks()
    if args.workload == "prefill":
        w = wl.RAGGED_PREFILL
        if args.batch:
            wl.RAGGED_PREFILL = wl.shrink(w, batch=args.batch)
        r = measure_prefill(args.seed, args.steps, args.warmup, peak_tf, head_dim=args.head_dim)
        wl.RAGGED_PREFILL = w
    elif args.workload == "prefill_variable_window":
        r = measure_prefill_fixed(args.seed, args.steps, args.warmup, peak_tf, variable_window=True)
    elif args.workload == "merge":
        r = measure_merge(args.seed, args.steps, args.warmup, peak_gbs, rows=args.batch or 8192)
    else:
        w = wl.DECODE_WORKLOADS[args.workload]
        if args.batch:
            pool = None if w.pool_pages is None else max(1000, w.pool_pages * args.batch // w.batch)
            wl.DECODE_WORKLOADS[args.workload] = wl.shrink(w, batch=args.batch, pool_pages=pool)
        dtype = torch.float16 if args.dtype == "f16" else torch.bfloat16
        r, _, _ = measure_workload(args.workload, args.seed, args.steps, args.warmup, peak_gbs,
                                   dtype=dtype)
        wl.DECODE_WORKLOADS[args.workload] = w
    torch.cuda.synchronize()
    emit({"profile_case": args.workload, "batch": args.batch, "plan": PLAN_OVERRIDES,
          "result": r})


def measured_peaks_all():
    """(HBM GB/s, bf16 TFLOP/s burst, source, bf16 TFLOP/s sustained or None)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return (d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured",
                d.get("bf16_tflops_sustained"))
    return 6800.0, 1900.0, "fallback", 1700.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


def kv_bytes(inp):
    """Algorithmic K+V bytes of one decode call: every visited key of every
    request, once per KV head, K and V, bf16 (window-trimmed, not page-rounded)."""
    seq = inp["seq_lens_kv"].cpu().tolist()
    if inp["qo_indptr"] is not None:
        ind = inp["qo_indptr"].cpu().tolist()
        qls = [ind[i + 1] - ind[i] for i in range(len(seq))]
    else:
        qls = [inp["q_len"]] * len(seq)
    W = inp["window_left"]
    D = inp["q"].shape[2]
    keys = 0
    for n, L in zip(seq, qls):
        first = max(0, n - L - W) if W >= 0 else 0
        keys += n - first
    return keys * inp["num_kv_heads"] * D * 2 * 2, keys


_ACTIVE_SAMPLER = None


def clock_mark(which):
    """Mark the start ("start") or end ("stop") of a timed region for the active
    ClockSampler, whose summary then keeps only the samples taken inside it."""
    if _ACTIVE_SAMPLER is not None:
        setattr(_ACTIVE_SAMPLER, "t_" + which, time.time())


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms; the summary keeps
    the samples stamped inside the timed region (clock_mark), or all of them if
    the region was too short to hold one."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t_start = self.t_stop = None

    def __enter__(self):
        global _ACTIVE_SAMPLER
        _ACTIVE_SAMPLER = self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        global _ACTIVE_SAMPLER
        if _ACTIVE_SAMPLER is self:
            _ACTIVE_SAMPLER = None
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    @staticmethod
    def _stamp(text):
        try:
            return datetime.datetime.strptime(text, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            try:
                samples.append((self._stamp(parts[0]), float(parts[1]), float(parts[2]),
                                {n for n, v in zip(names, parts[4:])
                                 if v.lower().startswith("active")}))
            except (ValueError, IndexError):
                continue
        window = "whole measurement"
        inside = samples
        if self.t_start is not None and self.t_stop is not None:
            inside = [x for x in samples
                      if x[0] is not None and self.t_start <= x[0] <= self.t_stop + 0.05]
            window = "timed region"
            if not inside:
                inside, window = samples, "whole measurement (timed region shorter than a sample)"
        if not inside:
            return None
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": inside[-1][2],
                "reasons": sorted(set().union(*(x[3] for x in inside))),
                "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg and the --impl reference arm)
# ---------------------------------------------------------------------------

def _oracle_task(task):
    """Run the fp64 oracle for one request in a worker process, repeating it
    until `min_seconds` have passed; return (seconds, repetitions)."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import oracle
    (q_bits, k_bits, v_bits, table, seq, L, Hkv, ps, causal, W, sinks, min_seconds) = task
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.paged_decode_request(0, q_bits, k_bits, v_bits, table[None], seq, 0, L, Hkv, ps,
                                    causal=causal, window_left=W, sinks=sinks)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            return el, reps


def oracle_sample_tasks(inp, n_requests, min_seconds=0.0):
    """Per-request oracle inputs (only the pages each request uses) for a sample;
    each task repeats its request for at least `min_seconds`.  Returns the tasks
    and the K+V bytes of one pass over each task's request."""
    import numpy as np
    import torch
    from paged_kv_attention_32_gb300 import workloads as wl
    seq = inp["seq_lens_kv"].cpu().numpy()
    bt = inp["block_tables"].cpu().numpy()
    ps = inp["page_size"]
    ind = (inp["qo_indptr"].cpu().numpy() if inp["qo_indptr"] is not None
           else np.arange(len(seq) + 1) * inp["q_len"])
    sinks = inp["sinks"].cpu().double().numpy() if inp["sinks"] is not None else None
    tasks, nbytes = [], []
    D = inp["q"].shape[2]
    for b in range(min(n_requests, len(seq))):
        n, L = int(seq[b]), int(ind[b + 1] - ind[b])
        npg = -(-n // ps)
        ids = torch.as_tensor(bt[b, :npg].astype(np.int64), device=inp["k_pages"].device)
        kb = wl.bf16_bits(inp["k_pages"].index_select(0, ids))
        vb = wl.bf16_bits(inp["v_pages"].index_select(0, ids))
        qb = wl.bf16_bits(inp["q"][int(ind[b]):int(ind[b + 1])])
        W = inp["window_left"]
        first = max(0, n - L - W) if W >= 0 else 0
        nbytes.append((n - first) * inp["num_kv_heads"] * D * 4)
        tasks.append((qb, kb, vb, np.arange(npg, dtype=np.int64), np.array([n]), L,
                      inp["num_kv_heads"], ps, inp["causal"], W, sinks, min_seconds))
    return tasks, nbytes


def run_oracle_sample(tasks, nbytes, cores):
    """Oracle over the sample on `cores` spawned worker processes (one task per
    worker).  Returns (bytes processed, makespan seconds)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_task, tasks, chunksize=1)
    loads = [0.0] * cores
    done = 0
    for (sec, reps), nb in sorted(zip(res, nbytes), key=lambda x: -x[0][0]):
        i = loads.index(min(loads))                # longest-first packing onto the cores
        loads[i] += sec
        done += reps * nb
    return done, max(loads)


def cpu_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


# ---------------------------------------------------------------------------
# GPU measurements
# ---------------------------------------------------------------------------

def make_plan(inp, **kw):
    from paged_kv_attention_32_gb300 import api
    args = dict(num_qo_heads=inp["q"].shape[1], num_kv_heads=inp["num_kv_heads"],
                page_size=inp["page_size"], max_pages_per_seq=inp["block_tables"].shape[1],
                num_pages=inp["k_pages"].shape[0], causal=inp["causal"],
                window_left=inp["window_left"], return_lse=inp["return_lse"],
                bmm2_scale=inp["bmm2_scale"])
    if inp["qo_indptr"] is not None:
        args["qo_indptr"] = inp["qo_indptr"].cpu()
    else:
        args["q_len"] = inp["q_len"]
    args.update(PLAN_OVERRIDES)
    args.update(kw)
    return api.paged_decode_plan(inp["seq_lens_kv"].cpu(), **args)


def decode_buffers(inp, plan):
    import torch
    q = inp["q"]
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=q.device)
    return out, lse, ws


def time_decode(inp, plan, steps, warmup, dist=None):
    """Device time per paged_decode_run call (CUDA events on the launching stream)."""
    import torch
    from paged_kv_attention_32_gb300 import api
    out, lse, ws = decode_buffers(inp, plan)
    stream = torch.cuda.current_stream()
    args = (plan, inp["q"], inp["k_pages"], inp["v_pages"], inp["block_tables"])
    kw = dict(seq_lens_kv=inp["seq_lens_kv"], sinks=inp["sinks"], out=out, lse=lse, workspace=ws,
              stream=stream)
    for _ in range(warmup):
        api.paged_decode_run(*args, **kw)
    torch.cuda.synchronize()
    plan.check()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clock_mark("start")
    e0.record(stream)
    for _ in range(steps):
        api.paged_decode_run(*args, **kw)
    e1.record(stream)
    torch.cuda.synchronize()
    clock_mark("stop")
    if dist is not None:
        dist.barrier()
    plan.check()
    return e0.elapsed_time(e1) / steps     # ms per call


def time_decode_e2e(inp, plan_kw, steps, warmup, in_place=True):
    """One serving step through the C ABI with host buffers, wall clock per step:
    ``paged_decode_step_host`` re-plans one plan on the step's host lengths, runs
    the decode on that step's q and block tables from pinned host memory and
    delivers O and the LSE to pinned host memory, then synchronises.  Staged, the
    step copies q / tables to device buffers first and O / LSE back after the
    run; ``in_place``, the kernels read q and the tables and write O and the LSE
    in the pinned host arrays themselves (the same bytes cross the host link,
    moved by the kernels' own loads and stores).  The KV pools are the cache:
    they stay resident on the device."""
    import torch
    from paged_kv_attention_32_gb300 import api
    q, bt, seq = inp["q"], inp["block_tables"], inp["seq_lens_kv"]
    rows = q.shape[:2]
    host = dict(
        q_host=q.cpu().pin_memory(), block_tables_host=bt.cpu().pin_memory(),
        seq_lens_kv_host=seq.cpu().pin_memory(),
        qo_indptr_host=None if inp["qo_indptr"] is None else inp["qo_indptr"].cpu().pin_memory(),
        out_host=torch.empty(q.shape, dtype=q.dtype).pin_memory(),
        lse_host=torch.empty(rows, dtype=torch.float32).pin_memory())
    if in_place:
        dev = dict(q_dev=host["q_host"], block_tables_dev=host["block_tables_host"],
                   seq_lens_kv_dev=host["seq_lens_kv_host"], out_dev=host["out_host"],
                   lse_dev=host["lse_host"])
    else:
        dev = dict(q_dev=torch.empty_like(q), block_tables_dev=torch.empty_like(bt),
                   seq_lens_kv_dev=torch.empty_like(seq), out_dev=torch.empty_like(q),
                   lse_dev=torch.empty(rows, dtype=torch.float32, device=q.device))
    io = api.DecodeHostIO(**host, **dev)
    t = io.tensors
    stream = torch.cuda.current_stream()
    bytes_in = q.numel() * q.element_size() + bt.numel() * 4 + seq.numel() * 4
    bytes_out = q.numel() * q.element_size() + (t["lse_host"].numel() * 4
                                                if inp["return_lse"] else 0)
    kw = dict(plan_kw)
    if t["qo_indptr_host"] is not None:
        kw["qo_indptr"] = t["qo_indptr_host"]
    plan = api.paged_decode_plan(t["seq_lens_kv_host"], stream=stream, **kw)   # re-planned per step

    step = api.DecodeStep(plan, io, inp["k_pages"], inp["v_pages"], sinks=inp["sinks"],
                          stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / steps
    plan.check()
    return ms, bytes_in, bytes_out


def reduce_over_ranks(ms, nbytes, dist=None, device="cpu"):
    """Whole-job figure of N replicas: the slowest rank's time and every rank's bytes
    (each rank decodes its own seeded batch, so the byte counts differ)."""
    if dist is None:
        return ms, nbytes
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    b = torch.tensor([float(nbytes)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(round(b.item()))


def headline_traffic(head):
    """DRAM bytes per headline launch from the ncu capture, scaled to this call's K+V bytes
    (None when the plan runs another kernel than the one captured)."""
    if KERNEL_SYMBOL[head["kernel"]] != NCU_TRAFFIC["kernel"]:
        return None
    return int(round(NCU_TRAFFIC["dram_bytes"] * head["kv_bytes"] / NCU_TRAFFIC["kv_bytes"]))


def measure_workload(name, seed, steps, warmup, peak_gbs, dist=None, dtype=None):
    """Inputs drawn on the GPU, plan, device timing; returns (result dict, inp, plan)."""
    import torch
    from paged_kv_attention_32_gb300 import workloads as wl
    w = wl.DECODE_WORKLOADS[name]
    inp = wl.make_decode_inputs(w, seed=seed, device="cuda", dtype=dtype or torch.bfloat16)
    plan = make_plan(inp, dtype=inp["q"].dtype)
    ms = time_decode(inp, plan, steps, warmup, dist)
    nbytes, keys = kv_bytes(inp)
    info = plan.info
    gbs = nbytes / (ms * 1e-3) / 1e9
    res = {"workload": w.name + (f" {inp['q'].dtype}" if dtype is not None else ""),
           "ms_per_call": round(ms, 5), "kv_bytes": nbytes,
           "kv_tokens": keys, "GB_per_s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak_gbs, 4),
           "kernel": ["cuda_core", "mma"][info["kernel"]], "ctas": info["num_items"],
           "split_requests": info["num_split"], "launches_per_call": 1}   # the split merge runs inside the decode kernel
    return res, inp, plan


def time_prefill_calls(run, steps, warmup):
    """Device time per call of `run` (CUDA events over `steps` back-to-back calls
    after `warmup`), with the SM clocks sampled during the timed calls."""
    import torch
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        clock_mark("start")
        e0.record()
        for _ in range(steps):
            run()
        e1.record()
        torch.cuda.synchronize()
        clock_mark("stop")
    return e0.elapsed_time(e1) / steps, clk.summary()


def prefill_result(name, ms, flops, peak_tflops, tiles, clocks):
    """A prefill line: achieved TFLOP/s against the measured bf16 peak taken as a
    burst (the main fraction) and as sustained under the power cap, with the
    clocks seen while timing (long runs of dense MMAs drive the part to its power
    cap, where the SM clock drops below its maximum)."""
    tf = flops / (ms * 1e-3) / 1e12
    _, _, _, sustained = measured_peaks_all()
    res = {"workload": name, "ms_per_call": round(ms, 4), "flops": flops,
           "TFLOP_per_s": round(tf, 1), "frac_of_measured_bf16": round(tf / peak_tflops, 4),
           "tiles": tiles, "clocks": clocks}
    if sustained:
        res["frac_of_measured_bf16_sustained"] = round(tf / sustained, 4)
    return res


def measure_prefill(seed, steps, warmup, peak_tflops, window_left=-1, dtype=None, head_dim=128,
                    cpu=False):
    """Ragged causal prefill; FLOPs = 4 * D per unmasked (query, key) pair per query head
    (with a window, row i of a request keeps min(i + 1, window_left + 1) keys).  With
    `cpu`, the fp64 oracle is timed beside it on a sample of the same inputs."""
    import torch
    from paged_kv_attention_32_gb300 import api
    from paged_kv_attention_32_gb300 import workloads as wl
    import dataclasses
    w = wl.RAGGED_PREFILL
    if head_dim != w.head_dim:
        w = dataclasses.replace(w, head_dim=head_dim, name=w.name.replace("D=128", f"D={head_dim}"))
    inp = wl.make_prefill_inputs(w, seed=seed, device="cuda")
    if dtype is not None:   # the same values drawn in bf16, held as fp16
        for key in ("q", "k", "v"):
            inp[key] = inp[key].to(dtype)
    lens = inp["lens"].tolist()
    if window_left >= 0:
        W1 = window_left + 1
        pairs = sum(min(n, W1) * (min(n, W1) + 1) // 2 + max(0, n - W1) * W1 for n in lens)
    else:
        pairs = sum(n * (n + 1) // 2 for n in lens)
    flops = 4 * head_dim * pairs * w.num_qo_heads
    name = w.name + (f" window_left={window_left}" if window_left >= 0 else "") + (
        f" {dtype}" if dtype is not None else "")
    try:
        plan = api.batch_prefill_plan(inp["qo_indptr"].cpu(), inp["kv_indptr"].cpu(),
                                      num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                                      window_left=window_left, dtype=inp["q"].dtype,
                                      head_dim=head_dim)
        out = torch.empty_like(inp["q"])
        ms, clocks = time_prefill_calls(
            lambda: api.batch_prefill_run(plan, inp["q"], inp["k"], inp["v"], out=out), steps,
            warmup)
        plan.check()
    except Exception as exc:   # reported, not hidden: the line says why there is no number
        return {"workload": name, "status": f"not measured: {exc}", "flops": flops}
    res = prefill_result(name, ms, flops, peak_tflops, plan.num_tiles, clocks)
    if cpu:
        res["cpu_baseline"] = prefill_cpu_baseline(inp, w)
    return res


def measure_prefill_fixed(seed, steps, warmup, peak_tflops, variable_window=False, dense=False):
    """Fixed-shape [B, S, H, D] prefill, B=4, S=4096, Hq=32, Hkv=8: causal, dense (every
    row sees every key), or variable_window with row i of each request seeing keys
    [s_i, i], s_i uniform in [max(0, i - 2047), i] (seeded).  FLOPs = 4 * D per visible
    (query, key) pair per head."""
    import numpy as np
    import torch
    from paged_kv_attention_32_gb300 import api
    B, S, Hq, Hkv = 4, 4096, 32, 8
    g = torch.Generator(device="cuda").manual_seed(seed + 7)
    q = torch.randn((B, S, Hq, 128), generator=g, device="cuda", dtype=torch.bfloat16)
    k = torch.randn((B, S, Hkv, 128), generator=g, device="cuda", dtype=torch.bfloat16)
    v = torch.randn((B, S, Hkv, 128), generator=g, device="cuda", dtype=torch.bfloat16)
    kw, name = {}, f"fixed-shape causal prefill B={B} S={S} Hq={Hq} Hkv={Hkv} D=128"
    pairs = B * S * (S + 1) // 2
    if dense:
        kw = dict(mask_type="dense")
        pairs = B * S * S
        name = f"fixed-shape dense prefill B={B} S={S} Hq={Hq} Hkv={Hkv} D=128"
    if variable_window:
        rng = np.random.default_rng(seed + 8)
        i = np.arange(S)
        st = (i - rng.integers(0, 2048, size=(B, S))).clip(0, None).astype(np.int32)
        en = np.tile(i, (B, 1)).astype(np.int32)
        kw = dict(mask_type="variable_window", variable_window_token_starts=st,
                  variable_window_token_ends=en)
        pairs = int((en - st + 1).sum())
        name = (f"fixed-shape variable_window prefill B={B} S={S} Hq={Hq} Hkv={Hkv} D=128, "
                "row i sees [i - U(0, 2047), i]")
    flops = 4 * 128 * pairs * Hq
    plan = api.batch_prefill_plan_fixed(B, S, S, num_qo_heads=Hq, num_kv_heads=Hkv, **kw)
    out = torch.empty_like(q)
    ms, clocks = time_prefill_calls(lambda: api.batch_prefill_run(plan, q, k, v, out=out), steps,
                                    warmup)
    plan.check()
    return prefill_result(name, ms, flops, peak_tflops, plan.num_tiles, clocks)


def measure_merge(seed, steps, warmup, peak_gbs, rows=8192):
    """Standalone attn_merge_lse: N=8 partial states of S=8192 rows (`rows`), H=32 heads,
    D=128 (fp32 V [N, S, H, D] and base-2 LSE [N, S, H]) merged into bf16 O and an fp32 LSE.
    Algorithmic bytes = every partial read once + the outputs written once."""
    import torch
    from paged_kv_attention_32_gb300 import api
    N, S, H, D = 8, rows, 32, 128
    g = torch.Generator(device="cuda").manual_seed(seed + 9)
    vs = torch.randn((N, S, H, D), generator=g, device="cuda", dtype=torch.float32)
    ss = torch.randn((N, S, H), generator=g, device="cuda", dtype=torch.float32)
    v_out = torch.empty((S, H, D), dtype=torch.bfloat16, device="cuda")
    s_out = torch.empty((S, H), dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        api.attn_merge_lse(vs, ss, v_out=v_out, s_out=s_out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        api.attn_merge_lse(vs, ss, v_out=v_out, s_out=s_out)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    nbytes = vs.numel() * 4 + ss.numel() * 4 + v_out.numel() * 2 + s_out.numel() * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"attn_merge_lse N={N} S={S} H={H} D={D} fp32 states -> bf16",
            "ms_per_call": round(ms, 5), "bytes": nbytes, "GB_per_s": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak_gbs, 4),
            "l2": "inputs (%.2f GB) larger than L2" % (vs.numel() * 4 / 1e9)}


def _oracle_worker(conn, task):
    """Long-lived oracle worker: holds one request's data, runs it on command."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    while True:
        msg = conn.recv()
        if msg is None:
            return
        conn.send(_oracle_task(task[:-1] + (msg,)))


class OraclePool:
    """One spawned process per sampled request (one per core); the request data
    is shipped once, then each `step(min_seconds)` runs every worker's request
    for at least that long.  Returns (bytes processed, makespan seconds)."""

    def __init__(self, tasks, nbytes):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        os.environ["OPENBLAS_NUM_THREADS"] = "1"
        os.environ["OMP_NUM_THREADS"] = "1"
        self.nbytes = nbytes
        self.procs, self.conns = [], []
        for t in tasks:
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(b, t), daemon=True)
            p.start()
            self.procs.append(p)
            self.conns.append(a)

    def step(self, min_seconds):
        for c in self.conns:
            c.send(min_seconds)
        res = [c.recv() for c in self.conns]
        done = sum(reps * nb for (sec, reps), nb in zip(res, self.nbytes))
        return done, max(sec for sec, _ in res)

    def close(self):
        for c in self.conns:
            c.send(None)
        for p in self.procs:
            p.join(timeout=10)


def cpu_baseline(inp, min_seconds=10.0):
    tasks, nbytes = oracle_sample_tasks(inp, cpu_cores())
    pool = OraclePool(tasks, nbytes)
    try:
        done, secs = pool.step(min_seconds)
    finally:
        pool.close()
    return {"value": round(done / secs / 1e9, 4), "unit": UNIT, "cores": len(tasks),
            "kind": "oracle",
            "sample": f"fp64 oracle, one spawned process per core, each repeating one of the "
                      f"first {len(tasks)} requests of the same batch for >= {min_seconds:.0f} s "
                      f"({done / 1e9:.2f} GB of K+V in {secs:.1f} s)"}


def _prefill_oracle_worker(conn, task):
    """Long-lived prefill oracle worker: one request's query rows of one GQA group,
    its keys and values for that group's KV head; repeats them on command."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import oracle
    q_bits, k_bits, v_bits, rows, flops = task
    lq, lk = q_bits.shape[0], k_bits.shape[0]
    ind_q, ind_k = [0, lq], [0, lk]
    while True:
        msg = conn.recv()
        if msg is None:
            return
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.prefill_request(0, q_bits, k_bits, v_bits, ind_q, ind_k, 1, causal=True,
                                   rows=rows)
            reps += 1
            el = time.perf_counter() - t0
            if el >= msg:
                break
        conn.send((el, reps * flops))


def prefill_cpu_baseline(inp, w, min_seconds=8.0, rows_per_task=32):
    """The fp64 oracle on the host cores, on a bounded sample of the ragged prefill:
    worker i takes request i % B and the query heads of KV head (i // B) % Hkv, and
    `rows_per_task` query rows spread evenly over the request; FLOPs = 4 * D per
    visible (row, key) pair per query head, as the GPU line counts them."""
    import multiprocessing as mp
    import numpy as np
    from paged_kv_attention_32_gb300 import workloads as wl
    ind = inp["qo_indptr"].cpu().numpy()
    B, G = len(ind) - 1, w.num_qo_heads // w.num_kv_heads
    ctx = mp.get_context("spawn")
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    procs, conns = [], []
    for i in range(cpu_cores()):
        b, hk = i % B, (i // B) % w.num_kv_heads
        s0, s1 = int(ind[b]), int(ind[b + 1])
        n = s1 - s0
        rows = np.unique(np.linspace(0, n - 1, min(rows_per_task, n)).astype(np.int64))
        flops = 4 * w.head_dim * G * int((rows + 1).sum())
        task = (wl.bf16_bits(inp["q"][s0:s1, hk * G:(hk + 1) * G]),
                wl.bf16_bits(inp["k"][s0:s1, hk:hk + 1]), wl.bf16_bits(inp["v"][s0:s1, hk:hk + 1]),
                rows, flops)
        a, c = ctx.Pipe()
        pr = ctx.Process(target=_prefill_oracle_worker, args=(c, task), daemon=True)
        pr.start()
        procs.append(pr)
        conns.append(a)
    try:
        for c in conns:
            c.send(min_seconds)
        res = [c.recv() for c in conns]
    finally:
        for c in conns:
            c.send(None)
        for pr in procs:
            pr.join(timeout=10)
    secs = max(r[0] for r in res)
    done = sum(r[1] for r in res)
    return {"value": round(done / secs / 1e12, 6), "unit": "TFLOP/s", "cores": len(procs),
            "kind": "oracle",
            "sample": f"fp64 oracle, one spawned process per core, each repeating {rows_per_task} "
                      f"causal rows of one request x the {G} query heads of one KV head for "
                      f">= {min_seconds:.0f} s ({done / 1e12:.3f} TFLOP in {secs:.1f} s)"}


def emit(line):
    print(json.dumps(line), flush=True)


def headline_config(w, inp, world):
    """The `config` object of the headline line, the same for both arms."""
    nbytes, keys = kv_bytes(inp)
    return {"workload": w.name, "batch": w.batch, "num_qo_heads": w.num_qo_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
            "kv_tokens": keys, "kv_bytes_per_call": nbytes,
            "l2": "inputs larger than L2 (each call reads >1 GB of K/V; no flush)",
            "parallelism": f"replicas x{world} (one batch per GPU)"}


def clocks_ok(clocks):
    """False when the clock record shows a throttle reason other than the power cap,
    or an SM clock well below its maximum with no reason given; None without a record."""
    if not clocks:
        return None
    bad = set(clocks.get("reasons", [])) - {"sw_power_cap"}
    low = clocks["sm_mhz"] < 0.85 * clocks["sm_max_mhz"] and not clocks.get("reasons")
    return not bad and not low


def compact(r):
    """A short summary of one sub-line (kept last on the JSON line, so that a reader
    keeping only the line's tail still sees every workload): ms per call, the achieved
    GB/s or TFLOP/s, the fraction of the measured peak, whether the clocks were clean,
    and the oracle's rate where one was timed."""
    if "status" in r:
        return {"status": r["status"][:60]}
    out = {"ms": float(f"{r.get('ms_per_call'):.4g}")}
    if "GB_per_s" in r:
        out.update(GBps=round(r["GB_per_s"]), frac=round(r.get("frac_of_measured_hbm"), 3))
    if "TFLOP_per_s" in r:
        out.update(TFLOPs=round(r["TFLOP_per_s"]), frac=round(r.get("frac_of_measured_bf16"), 3))
    if "clocks" in r:
        out["clk"] = clocks_ok(r["clocks"])
    if r.get("cpu_baseline"):
        out["oracle"] = r["cpu_baseline"]["value"]
    return out


def reference_arm(args, rank):
    """--impl reference: the fp64 CPU oracle timed on the host cores."""
    if rank != 0:
        return
    from paged_kv_attention_32_gb300 import workloads as wl
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = wl.make_decode_inputs(wl.DECODE_WORKLOADS[HEADLINE], seed=args.seed, device=dev)
    tasks, nbytes = oracle_sample_tasks(inp, cpu_cores())
    cores = len(tasks)
    # each step: every core runs its sampled request for a slice of a ~90 s budget
    per_step = max(0.05, min(2.0, 90.0 / max(1, args.steps + args.warmup)))
    pool = OraclePool(tasks, nbytes)
    try:
        for _ in range(args.warmup):
            pool.step(per_step)
        runs = [pool.step(per_step) for _ in range(args.steps)]
    finally:
        pool.close()
    total = sum(s for _, s in runs)
    value = sum(d for d, _ in runs) / total / 1e9
    cpu = {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"fp64 oracle, one spawned process per core, each repeating one of the "
                     f"first {cores} requests of the {wl.DECODE_WORKLOADS[HEADLINE].name} batch "
                     f"for >= {per_step:.2f} s per step"}
    emit({"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
          "ms_per_step": round(total * 1e3 / args.steps, 2), "higher_is_better": True,
          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
          "config": headline_config(wl.DECODE_WORKLOADS[HEADLINE], inp,
                                    int(os.environ.get("WORLD_SIZE", "1"))),
          "cpu_baseline": cpu,
          "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}})


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = tdist
    if args.impl == "reference":
        reference_arm(args, rank)
        if dist is not None:
            dist.destroy_process_group()
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the CUDA path (no CPU fallback)")
    torch.cuda.set_device(local)
    if args.mma_min_rows:
        PLAN_OVERRIDES["mma_min_rows"] = args.mma_min_rows
    if args.split_waves:
        PLAN_OVERRIDES["split_waves"] = args.split_waves
    if args.workload is not None:
        profile_case(args)
        return
    peak_gbs, peak_tf, peak_kind = measured_peaks()

    # ---- headline: Llama-3-8B-shaped decode ----
    with ClockSampler(local) as clk:
        head, inp, plan = measure_workload(HEADLINE, args.seed + rank, args.steps, args.warmup,
                                           peak_gbs, dist)
    clocks = clk.summary()
    ms, total_bytes = reduce_over_ranks(head["ms_per_call"], head["kv_bytes"], dist, "cuda")
    value = total_bytes / (ms * 1e-3) / 1e9
    gbs_kernel = head["kv_bytes"] / (head["ms_per_call"] * 1e-3) / 1e9

    # end to end through the public API on every rank: slowest rank, all ranks' bytes
    from paged_kv_attention_32_gb300 import workloads as wl
    w = wl.DECODE_WORKLOADS[HEADLINE]
    plan_kw = dict(num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                   page_size=w.page_size, max_pages_per_seq=inp["block_tables"].shape[1],
                   num_pages=inp["k_pages"].shape[0], return_lse=w.return_lse, q_len=1)
    if dist is not None:
        dist.barrier()
    e2e_ms, bin_, bout = time_decode_e2e(inp, plan_kw, min(args.steps, 50),
                                         max(3, min(args.warmup, 3)))
    e2e_ms, e2e_bytes = reduce_over_ranks(e2e_ms, head["kv_bytes"], dist, "cuda")
    staged_ms, _, _ = time_decode_e2e(inp, plan_kw, min(args.steps, 50),
                                      max(3, min(args.warmup, 3)), in_place=False)
    staged_ms, _ = reduce_over_ranks(staged_ms, head["kv_bytes"], dist, "cuda")

    line = None
    if rank == 0:
        e2e_val = e2e_bytes / (e2e_ms * 1e-3) / 1e9
        cpu = cpu_baseline(inp) if (world == 1 and not args.no_cpu) else None
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": headline_config(w, inp, world),
            "roofline": {"bound": "hbm", "kernel": KERNEL_SYMBOL[head["kernel"]],
                         "achieved": round(gbs_kernel, 1), "peak": peak_gbs, "unit": "GB/s",
                         "frac": round(gbs_kernel / peak_gbs, 4), "peak_source": peak_kind,
                         "traffic": headline_traffic(head)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_val, 1), "unit": UNIT, "ms_per_step": round(e2e_ms, 4),
                    "h2d_bytes_per_step": bin_, "d2h_bytes_per_step": bout,
                    "note": "paged_decode_step_host per step: host re-planning of one plan "
                            "on the step's lengths, run with q/tables read and O/LSE written "
                            "by the kernels in place in pinned host memory (NVLink-C2C), "
                            "synchronise; the KV cache stays resident",
                    "staged": {"value": round(e2e_bytes / (staged_ms * 1e-3) / 1e9, 1),
                               "ms_per_step": round(staged_ms, 4),
                               "note": "same step with device staging: pinned H2D of q/tables "
                                       "(queued before the re-plan), run, D2H of O and LSE"}},
            "gpu_launches": args.steps * head["launches_per_call"],
            "clocks": clocks,
        }
    del inp, plan
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_extra:
        extra = {}
        for name in ("tiny", "skewed", "spec"):
            r, i2, p2 = measure_workload(name, args.seed, max(5, args.steps // 2),
                                         max(3, args.warmup), peak_gbs)
            extra[name] = r
            del i2, p2
            torch.cuda.empty_cache()
        extra["prefill"] = measure_prefill(args.seed, max(3, args.steps // 4), 3, peak_tf,
                                           cpu=world == 1 and not args.no_cpu)
        extra["prefill_window"] = measure_prefill(args.seed, max(3, args.steps // 4), 3, peak_tf,
                                                  window_left=PREFILL_WINDOW)
        extra["prefill_fixed"] = measure_prefill_fixed(args.seed, max(3, args.steps // 4), 3,
                                                       peak_tf)
        r16, i16, p16 = measure_workload(HEADLINE, args.seed, max(5, args.steps // 2),
                                         max(3, args.warmup), peak_gbs, dtype=torch.float16)
        extra["llama3_8b_f16"] = r16
        del i16, p16
        torch.cuda.empty_cache()
        extra["prefill_f16"] = measure_prefill(args.seed, max(3, args.steps // 4), 3, peak_tf,
                                               dtype=torch.float16)
        extra["prefill_d256"] = measure_prefill(args.seed, max(3, args.steps // 4), 3, peak_tf,
                                                head_dim=256)
        extra["prefill_variable_window"] = measure_prefill_fixed(
            args.seed, max(3, args.steps // 4), 3, peak_tf, variable_window=True)
        extra["prefill_fixed_dense"] = measure_prefill_fixed(
            args.seed, max(3, args.steps // 4), 3, peak_tf, dense=True)
        extra["merge_lse"] = measure_merge(args.seed, max(5, args.steps // 2), max(3, args.warmup),
                                           peak_gbs)
        line["decode_headline"] = head
        line["other_workloads"] = extra
        # last key: one short entry per workload, so the line's tail names them all
        per = {"llama3_8b": compact(dict(head, clocks=clocks))}
        per.update((k, compact(v)) for k, v in extra.items())
        if cpu is not None:
            per["llama3_8b"]["oracle"] = cpu["value"]
        line["per_config"] = per
    if rank == 0:
        emit(line)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
