"""Benchmark: paged decode attention KV GB/s and sequences/s on one GB300.

One step = one decode step of one attention layer for the whole batch:
pkv_append of every sequence's new token (K/V scatter) followed by
pkv_decode_attention (split-KV decode + LSE combine), all through the C ABI.

Default workload: the 70B-class GQA decode batch (B=64, H_q=64, H_kv=8,
d_head=128, 16-token blocks, context ~ U[512, 8192], bf16 KV; about 1.14 GB of
K/V read per step, far larger than the 129 MB L2, so no flush is needed).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--split-tokens T]

Prints one JSON line.  value = KV bytes attended per step * steps / time
(GB/s, 1e9 bytes), whole job over all ranks.  With --gpus N > 1 (torchrun)
each rank runs an independent replica on its own GPU (the path has no
exchange step); value sums the ranks' bytes over the slowest rank's time.

--impl reference times the float64 CPU oracle (the reference of this
library) on the host cores over a bounded sample of the same workload.

--op cascade | multi_query | block_copy | host_swap times one of the other
hot-path operations instead of the decode step (one JSON line with "op"):
cascade decode on the shared-prefix workload (prefix kernel against the bf16
tensor peak), multi-token query attention on the GQA workload (--q-len new
tokens per sequence), the copy-on-write block copy (HBM), and block moves
between HBM and pinned host memory (against a contiguous copy over the same
link).
"""

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV GB/s & seqs/s at 1 GB300; fraction of HBM roofline"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000  # GB300 L2 (the flush writes twice this)
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None,
                    help="default: gqa_bf16 (shared_prefix for --op cascade)")
    ap.add_argument("--op", default="decode",
                    choices=["decode", "cascade", "multi_query", "block_copy", "host_swap"],
                    help="decode (the headline step) or one of the other hot-path operations")
    ap.add_argument("--q-len", type=int, default=4, help="new tokens per sequence for --op multi_query")
    ap.add_argument("--split-tokens", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.workload is None:
        args.workload = "shared_prefix" if args.op == "cascade" else "gqa_bf16"
    return args


# ---------------------------------------------------------------- oracle leg

def _oracle_unit_worker(args):
    """Oracle decode of one (sequence, KV head) unit on its own blocks;
    returns (seconds, (b, h), output [G, D])."""
    import numpy as np
    from oracle import paged_attention as PA
    key, q_bits, k_blocks, v_blocks, kind, ks, vs, ctx, bs, scale = args
    n = k_blocks.shape[0]
    table = np.arange(n, dtype=np.int32)[None, :]
    t0 = time.perf_counter()
    if kind == "e4m3":
        out = PA.decode_attention(q_bits[None], k_blocks, v_blocks, PA.E4M3, table, np.array([ctx]), scale,
                                  np.array([[ks]], dtype=np.float32), np.array([[vs]], dtype=np.float32))
    else:
        out = PA.decode_attention(q_bits[None], k_blocks, v_blocks, PA.BF16, table, np.array([ctx]), scale)
    return time.perf_counter() - t0, key, out[0]


def _unit_payload(case, b, h, ctx_attended):
    import torch
    from tests.gpu_support import bits16, bytes8
    G = case["H_q"] // case["H_kv"]
    n = -(-ctx_attended // case["bs"])
    ids = case["block_tables"][b, :n].to(torch.int64).to(case["k_cache"].device)
    raw = bytes8 if case["kv"] == "e4m3" else bits16
    kb = raw(case["k_cache"][ids][:, h:h + 1])
    vb = raw(case["v_cache"][ids][:, h:h + 1])
    q = bits16(case["q"][0, b, h * G:(h + 1) * G])
    ks = vs = None
    if case["kv"] == "e4m3":
        ks = float(case["k_scale"][b, h])
        vs = float(case["v_scale"][b, h])
    return ((b, h), q, kb, vb, case["kv"], ks, vs, ctx_attended, case["bs"], case["scale"])


def oracle_throughput(case, seconds, order_seed=0, return_outputs=False):
    """Run the oracle over (sequence, KV head) units in a spawn process pool,
    one single-threaded process per host core, until `seconds` of wall time
    are used.  Returns (GB/s of KV attended, units done, processes, wall
    seconds[, {(b, h): oracle output [G, D]}])."""
    import multiprocessing as mp
    import numpy as np
    cores = len(os.sched_getaffinity(0))
    procs = max(1, min(cores, 32))
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    rng = np.random.default_rng(order_seed)
    units = [(b, h) for b in range(case["B"]) for h in range(case["H_kv"])]
    rng.shuffle(units)
    ctx = (case["ctx"] + 1).tolist()
    per_unit_bytes = lambda b: ctx[b] * case["D"] * 2 * 2
    ctxm = mp.get_context("spawn")
    done_bytes = 0
    done = 0
    outputs = {}
    with ctxm.Pool(procs) as pool:
        # warm the workers (imports) before timing
        pool.map(_noop, range(procs))
        t0 = time.perf_counter()
        i = 0
        while i < len(units) and time.perf_counter() - t0 < seconds:
            batch = units[i:i + procs]
            payloads = [_unit_payload(case, b, h, ctx[b]) for b, h in batch]
            for _, key, out in pool.map(_oracle_unit_worker, payloads):
                outputs[key] = out
            done_bytes += sum(per_unit_bytes(b) for b, _ in batch)
            done += len(batch)
            i += procs
        wall = time.perf_counter() - t0
    throughput_gbs = done_bytes / wall / 1e9
    if return_outputs:
        return throughput_gbs, done, procs, wall, outputs
    return throughput_gbs, done, procs, wall


def _oracle_mq_unit_worker(args):
    """Oracle multi-token attention of one (sequence, KV head) unit; returns
    (seconds, (b, h), output [q_len, G, D])."""
    import numpy as np
    from oracle import paged_attention as PA
    key, q_bits, k_blocks, v_blocks, ctx, scale = args
    table = np.arange(k_blocks.shape[0], dtype=np.int32)[None, :]
    t0 = time.perf_counter()
    out = PA.multi_query_attention(q_bits[None], k_blocks, v_blocks, PA.BF16, table, np.array([ctx]), scale)
    return time.perf_counter() - t0, key, out[0]


def oracle_mq_throughput(case, q, lens, seconds):
    """The oracle's multi-token attention over (sequence, KV head) units of
    q [B, q_len, H_q, D] against the cache as it is, lens [B] tokens each
    (the new ones included), in a spawn pool of one process per host core,
    until `seconds` of wall time are used.  Returns (KV GB/s, units,
    processes, wall seconds, {(b, h): output [q_len, G, D]})."""
    import multiprocessing as mp
    import numpy as np
    import torch
    from tests.gpu_support import bits16
    cores = len(os.sched_getaffinity(0))
    procs = max(1, min(cores, 32))
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    G = case["H_q"] // case["H_kv"]
    units = [(b, h) for b in range(case["B"]) for h in range(case["H_kv"])]
    np.random.default_rng(1).shuffle(units)
    L = lens.cpu().tolist()
    qb = bits16(q)

    def payload(b, h):
        n = -(-L[b] // case["bs"])
        ids = case["block_tables"][b, :n].to(torch.int64).to(case["k_cache"].device)
        return ((b, h), qb[b, :, h * G:(h + 1) * G], bits16(case["k_cache"][ids][:, h:h + 1]),
                bits16(case["v_cache"][ids][:, h:h + 1]), L[b], case["scale"])

    done_bytes, done, outputs = 0, 0, {}
    with mp.get_context("spawn").Pool(procs) as pool:
        pool.map(_noop, range(procs))
        t0 = time.perf_counter()
        i = 0
        while i < len(units) and time.perf_counter() - t0 < seconds:
            batch = units[i:i + procs]
            for _, key, out in pool.map(_oracle_mq_unit_worker, [payload(b, h) for b, h in batch]):
                outputs[key] = out
            done_bytes += sum(L[b] * case["D"] * 4 for b, _ in batch)
            done += len(batch)
            i += procs
        wall = time.perf_counter() - t0
    return done_bytes / wall / 1e9, done, procs, wall, outputs


def _noop(_):
    import numpy  # noqa: F401
    from oracle import paged_attention  # noqa: F401
    return 0


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()

    def summary(self, t_begin, t_end):
        rows = []
        try:
            with open(self.file.name) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    except ValueError:
                        continue
                    rows.append((ts, parts))
        finally:
            os.unlink(self.file.name)
        inside = [p for ts, p in rows if t_begin - 0.05 <= ts <= t_end + 0.05]
        use = inside if inside else [p for _, p in rows]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(p[2]) for p in use if p[2].replace(".", "").isdigit()]
        smax = [float(p[3]) for p in use if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in use for n, v in zip(names, p[6:10]) if v.lower() == "active"})
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
               "samples": len(use), "samples_in_timed_region": len(inside)}
        pw = [float(p[4]) for p in use if p[4].replace(".", "").isdigit()]
        if pw:
            out["power_w_max"] = max(pw)
        return out


# ---------------------------------------------------------------- helpers

def max_over_ranks(x, device="cpu"):
    """Largest value of x over all ranks (x itself with one process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step, steps, world, slowest_ms):
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return bytes_per_rank_step * steps * world / (slowest_ms / 1e3) / 1e9


def replica_seed(base_seed, rank):
    """Each replica draws its own workload (same shapes, different values)."""
    return base_seed + 1000 * rank


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense bf16 tensor peak (burst: kernels timed on their own)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("decode.cu", "decode_common.cuh", "pkv_device.cuh", "pkv_internal.h"):
        with open(os.path.join(ROOT, "paged_kv_cache_222_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, split_tokens):
    """DRAM bytes per launch of the split kernel from a committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "decode_split_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    for r in rec.get("records", []):
        if r.get("workload") == workload and r.get("kernel_src") == kernel_source_hash():
            return r.get("dram_bytes_per_launch_full")
    return None


def workload_config(case, args, kv_bytes, plan):
    ctx = case["ctx"]
    cfg = {"workload": args.workload, "B": case["B"], "H_q": case["H_q"], "H_kv": case["H_kv"],
           "d_head": case["D"], "block_size": case["bs"], "kv_dtype": case["kv"],
           "context_attended": f"{int(ctx.min()) + 1}..{int(ctx.max()) + 1} (mean {float(ctx.float().mean()) + 1:.0f})",
           "kv_bytes_per_step": kv_bytes,
           "split": ("balanced ranges over %d warps" % plan.workers) if plan.mode == 0
                    else ("%d tokens x %d splits" % (plan.split_tokens, plan.max_splits)),
           "l2": "inputs larger than L2 (no flush)" if kv_bytes > L2_BYTES else
                 "L2 flushed between steps (258 MB write outside each step's events)",
           "parallelism": "replicas"}
    return cfg


# ---------------------------------------------------------------- arms

def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is a bounded sample of
    the workload's (sequence, KV head) units."""
    if rank != 0:
        return
    import workloads as W
    case = W.make_case(args.workload, device="cpu")
    per_step = max(2.0, min(8.0, 120.0 / max(1, args.steps + args.warmup)))
    vals = []
    cores = None
    units = 0
    for s in range(args.warmup + args.steps):
        gbs, n, procs, wall = oracle_throughput(case, per_step, order_seed=s)
        cores = procs
        if s >= args.warmup:
            vals.append(gbs)
            units += n
    value = statistics.median(vals) if vals else 0.0
    kv_bytes = int(((case["ctx"] + 1).to(float) * case["H_kv"] * case["D"] * 4).sum())
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": kv_bytes / (value * 1e9) * 1e3 if value else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.workload, "B": case["B"], "H_q": case["H_q"], "H_kv": case["H_kv"],
                       "d_head": case["D"], "block_size": case["bs"], "kv_bytes_per_step": kv_bytes},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{units} (sequence, KV head) units over {args.steps} steps of "
                                       f"~{per_step:.0f} s each; float64 numpy oracle, one process per core"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_cache_222_gb300 as pkv
    import workloads as W
    from paged_kv_cache_222_gb300 import build

    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
    spec = W.spec(args.workload)
    spec["seed"] = replica_seed(spec["seed"], rank)
    case = W.make_case(spec, device=dev)
    B, bs = case["B"], case["bs"]
    fp8 = case["kv"] == "e4m3"
    if fp8:
        from tests.gpu_support import fill_fp8_cache
        fill_fp8_cache(case)
    bt = case["block_tables"].to(dev)
    ctx = case["ctx"].to(dev)
    lens = (ctx + 1).to(torch.int32)
    max_len = int(case["ctx"].max()) + 1
    slots = pkv.slots_for_positions(bt, torch.arange(B, device=dev), ctx.to(torch.int64), bs)
    q = case["q"][0].contiguous()
    kn = case["k_new"][0].contiguous()
    vn = case["v_new"][0].contiguous()
    ks = case.get("k_scale") if fp8 else None
    vs = case.get("v_scale") if fp8 else None
    out = torch.empty((B, case["H_q"], case["D"]), dtype=torch.float32, device=dev)
    plan = pkv.decode_plan(B, case["H_q"], case["k_cache"], max_len, args.split_tokens)
    ws = torch.empty(max(1, int(plan.workspace_bytes)), dtype=torch.uint8, device=dev)
    esz = 1 if fp8 else 2
    kv_bytes = int(((case["ctx"] + 1).to(torch.float64) * case["H_kv"] * case["D"] * 2 * esz).sum())

    def step():
        pkv.append(kn, vn, slots, case["k_cache"], case["v_cache"], ks, vs)
        pkv.decode_attention(q, case["k_cache"], case["v_cache"], bt, lens, case["scale"], ks, vs,
                             max_context_len=max_len, out=out, split_tokens=args.split_tokens,
                             workspace=ws)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if pkv.device_error(dev) != 0:
        raise RuntimeError("device error during warm-up")

    # inputs that fit in L2 are timed step by step with L2 flushed in between
    # (a write of twice the L2 size outside each step's events)
    flush = kv_bytes <= L2_BYTES
    scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None
    clocks = ClockSampler(local_rank)
    clocks.start()
    barrier()
    t_wall0 = time.time()
    if flush:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            scrub.zero_()
            a.record(stream)
            step()
            b.record(stream)
    else:
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
    barrier()
    t_wall1 = time.time()
    clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in evs) if flush else ev0.elapsed_time(ev1)
    clk = clocks.summary(t_wall0, t_wall1)

    # the same steps again with every library launch bracketed by CUDA events
    # on its own stream: per-kernel device times (event records sit between
    # the kernels, so this pass is not the one `value` comes from)
    pkv.trace_read()
    pkv.trace_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    pkv.trace_enable(False)
    trace = pkv.trace_read()

    ms_max = max_over_ranks(ms, dev)
    value = job_throughput(kv_bytes, args.steps, world, ms_max)
    seqs = B * args.steps * world / (ms_max / 1e3)

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs from pinned host memory and reads its output back, as
    # a serving loop does: the copies run on a copy stream into two sets of
    # device buffers, one step ahead of the compute (step i+1's inputs move
    # while step i computes; step i's output moves back while step i+1
    # computes); the timed region spans all of them.
    pin = lambda t: t.cpu().pin_memory()
    h_in = [pin(t) for t in (q, kn, vn, slots, bt, lens)]
    h_outs = [torch.empty(out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    d_in = [[torch.empty_like(t) for t in (q, kn, vn, slots, bt, lens)] for _ in range(2)]
    d_out = [torch.empty_like(out) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    e2e_steps = max(3, min(args.steps, 500))
    cstream = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]

    def h2d_copy(i):  # on the copy stream
        if i >= 2:
            cstream.wait_event(ev_done[i % 2])     # step i-2 is done with this set
        for d, h in zip(d_in[i % 2], h_in):
            d.copy_(h, non_blocking=True)
        ev_in[i % 2].record(cstream)

    def e2e_run(n):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        cstream.wait_event(start)
        with torch.cuda.stream(cstream):
            h2d_copy(0)
        for i in range(n):
            if i + 1 < n:
                with torch.cuda.stream(cstream):
                    h2d_copy(i + 1)
            stream.wait_event(ev_in[i % 2])
            d_q, d_kn, d_vn, d_slots, d_bt, d_lens = d_in[i % 2]
            pkv.append(d_kn, d_vn, d_slots, case["k_cache"], case["v_cache"], ks, vs)
            pkv.decode_attention(d_q, case["k_cache"], case["v_cache"], d_bt, d_lens, case["scale"], ks, vs,
                                 max_context_len=max_len, out=d_out[i % 2], split_tokens=args.split_tokens,
                                 workspace=ws)
            ev_done[i % 2].record(stream)
            with torch.cuda.stream(cstream):
                cstream.wait_event(ev_done[i % 2])
                h_outs[i % 2].copy_(d_out[i % 2], non_blocking=True)
        tail = torch.cuda.Event()
        tail.record(cstream)
        stream.wait_event(tail)
        end.record(stream)
        return start, end

    e2e_run(3)
    barrier()
    e0, e1 = e2e_run(e2e_steps)
    barrier()
    e2e_value = job_throughput(kv_bytes, e2e_steps, world, max_over_ranks(e0.elapsed_time(e1), dev))
    if pkv.device_error(dev) != 0:
        raise RuntimeError("device error during the timed region")

    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    split = trace.get("decode_split", (0, 0.0))
    avg_ms = split[1] / split[0] if split[0] else float("nan")
    achieved = kv_bytes / (avg_ms / 1e3) / 1e9 if split[0] else None
    launches = sum(n for n, _ in trace.values())   # per traced pass of args.steps steps
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if not fp8 else "e4m3",
        "data": "synthetic",
        "config": workload_config(case, args, kv_bytes, plan),
        "seqs_per_s": seqs,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": (achieved / peak) if achieved else None,
                     "peak_source": f"{peak_kind} (hbm_gbs, copy bandwidth)",
                     "kernel": "decode_split", "algorithmic_bytes_per_launch": kv_bytes,
                     "avg_launch_ms": avg_ms,
                     "traffic": recorded_traffic(args.workload, args.split_tokens)},
        "kernel_times_ms": {k: {"launches": n, "avg_ms": t / n} for k, (n, t) in trace.items()},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps},
        "clocks": clk,
        "gpu_launches": launches,
    }
    if case.get("prefix", 0):
        # sequences sharing their first blocks: those bytes counted once, each
        # private suffix once (same time base as `value`)
        esz = 1 if fp8 else 2
        uniq = (case["prefix"] + float((case["ctx"].double() + 1 - case["prefix"]).sum())) * \
            case["H_kv"] * case["D"] * 2 * esz
        line["unique_GBs"] = value * uniq / kv_bytes
    if not args.no_cpu_baseline and world == 1:
        gbs, n, procs, wall, ref = oracle_throughput(case, args.cpu_seconds, return_outputs=True)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": procs, "kind": "oracle",
                                "sample": f"{n} of {B * case['H_kv']} (sequence, KV head) units of the "
                                          f"{args.workload} step, {wall:.1f} s wall, float64 numpy, "
                                          f"one process per core"}
        # the timed steps' output against the oracle on the same units
        got = out.cpu().numpy()
        G = case["H_q"] // case["H_kv"]
        err = max((float(abs(got[b, h * G:(h + 1) * G] - o).max()) for (b, h), o in ref.items()), default=None)
        line["parity"] = {"max_abs_err": err, "units": len(ref), "tolerance": 5e-3 if fp8 else 2e-3}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- other operations

def _time_on_stream(fn, steps, warmup, stream, sync):
    import torch
    for _ in range(max(3, warmup)):
        fn()
    sync()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    sync()
    return e0.elapsed_time(e1) / steps


def _traced(pkv, fn, steps, sync):
    pkv.trace_read()
    pkv.trace_enable(True)
    for _ in range(steps):
        fn()
    sync()
    pkv.trace_enable(False)
    return {k: (n, t) for k, (n, t) in pkv.trace_read().items()}


def run_op(args, local_rank):
    """One JSON line for a hot-path operation other than the decode step
    (cascade decode, multi-token query, block copy, host swap); device-timed
    with CUDA events on the launching stream, per-kernel times from the
    library's trace."""
    import numpy as np
    import torch
    import paged_kv_cache_222_gb300 as pkv
    import workloads as W
    from paged_kv_cache_222_gb300 import build

    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sync = lambda: torch.cuda.synchronize(dev)
    hbm, hbm_kind = measured_peaks()
    tf_peak, tf_kind = measured_bf16_tflops()
    steps, warm = args.steps, args.warmup
    line = {"op": args.op, "n_gpus": 1, "steps": steps, "warmup": warm, "data": "synthetic"}

    if args.op == "cascade":
        case = W.make_case(args.workload, device=dev)
        B, bs, prefix = case["B"], case["bs"], case["prefix"]
        bt = case["block_tables"].to(dev)
        lens = (case["ctx"] + 1).to(dev).to(torch.int32)
        mx = int(lens.max())
        q = case["q"][0].contiguous()
        out = torch.empty((B, case["H_q"], case["D"]), device=dev)
        pblocks = bt[0, :prefix // bs].contiguous()
        plan = pkv.cascade_plan(B, case["H_q"], case["k_cache"], prefix, mx)
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
        fn = lambda: pkv.cascade_decode_attention(q, case["k_cache"], case["v_cache"], pblocks, prefix, bt, lens,
                                                  case["scale"], mx, out=out, workspace=ws)
        plain = lambda: pkv.decode_attention(q, case["k_cache"], case["v_cache"], bt, lens, case["scale"],
                                             max_context_len=mx, out=out)
        ms = _time_on_stream(fn, steps, warm, stream, sync)
        ms_plain = _time_on_stream(plain, steps, warm, stream, sync)
        tr = _traced(pkv, fn, steps, sync)
        logical = float((case["ctx"].double() + 1).sum()) * case["H_kv"] * case["D"] * 4
        unique = (prefix + float((case["ctx"].double() + 1 - prefix).sum())) * case["H_kv"] * case["D"] * 4
        n, t = tr.get("cascade_prefix", (0, 0.0))
        pf_ms = t / n if n else float("nan")
        n2, t2 = tr.get("decode_split", (0, 0.0))
        sf_ms = t2 / n2 if n2 else float("nan")
        flops = 4.0 * B * case["H_q"] * prefix * case["D"]
        achieved = flops / (pf_ms / 1e3) / 1e12
        suffix_bytes = float((case["ctx"].double() + 1 - prefix).sum()) * case["H_kv"] * case["D"] * 4
        sf_gbs = suffix_bytes / (sf_ms / 1e3) / 1e9
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        row_blocks = -(-B * (case["H_q"] // case["H_kv"]) // 256) * case["H_kv"]
        sm_share = min(1.0, row_blocks * plan.workers / sms)   # SMs the prefix CTAs hold (one per SM)
        prefix_line = {"bound": "tensor", "kernel": "cascade_prefix", "achieved": achieved, "peak": tf_peak,
                       "unit": "TFLOP/s", "frac": achieved / tf_peak,
                       "peak_source": f"{tf_kind} (bf16_tflops, burst)", "algorithmic_flops_per_launch": flops,
                       "avg_launch_ms": pf_ms, "sm_share": sm_share,
                       "frac_of_its_sms": achieved / (tf_peak * sm_share), "traffic": None}
        suffix_line = {"bound": "hbm", "kernel": "decode_split (suffixes, beside the prefix)", "achieved": sf_gbs,
                       "peak": hbm, "unit": "GB/s", "frac": sf_gbs / hbm,
                       "peak_source": f"{hbm_kind} (hbm_gbs, copy bandwidth)",
                       "algorithmic_bytes_per_launch": suffix_bytes, "avg_launch_ms": sf_ms, "traffic": None}
        # the roofline line is the kernel that holds more SM time (its duration
        # times the SMs it runs on: the prefix CTAs hold sm_share of them, the
        # suffix decode the rest); the other rides along
        pf_smt, sf_smt = pf_ms * sm_share, sf_ms * (1.0 - sm_share)
        dominant, other = (prefix_line, suffix_line) if pf_smt > sf_smt else (suffix_line, prefix_line)
        line.update({"metric": "cascade decode KV GB/s (logical bytes: every sequence's whole context)",
                     "value": logical / ms / 1e6, "unit": "GB/s", "ms_per_step": ms, "higher_is_better": True,
                     "dtype": "bf16", "unique_GBs": unique / ms / 1e6, "plain_decode_ms": ms_plain,
                     "config": {"workload": args.workload, "B": B, "H_q": case["H_q"], "H_kv": case["H_kv"],
                                "d_head": case["D"], "block_size": bs, "shared_prefix": prefix,
                                "prefix_ranges": plan.workers, "prefix_range_tokens": plan.prefix_split_tokens,
                                "suffix_split_tokens": plan.split_tokens},
                     "kernel_times_ms": {k: {"launches": nn, "avg_ms": tt / nn} for k, (nn, tt) in tr.items() if nn},
                     "roofline": dominant, "roofline_other_kernel": other})
        if not args.no_cpu_baseline:
            # the oracle (plain decode of every sequence's whole context; the
            # cascade reaches the same result) on (sequence, KV head) units
            gbs, nu, procs, wall, ref = oracle_throughput(case, args.cpu_seconds, return_outputs=True)
            got = out.cpu().numpy()
            G = case["H_q"] // case["H_kv"]
            err = max(float(np.abs(got[b, h * G:(h + 1) * G] - r).max()) for (b, h), r in ref.items())
            line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": procs, "kind": "oracle",
                                    "sample": f"{nu} of {B * case['H_kv']} (sequence, KV head) units, "
                                              f"{wall:.1f} s wall, float64 numpy, one process per core"}
            line["parity"] = {"max_abs_err": err, "units": nu, "tolerance": 2e-3}
    elif args.op == "multi_query":
        ql = args.q_len
        case = W.make_case(args.workload, device=dev, steps=ql)
        B = case["B"]
        bt = case["block_tables"].to(dev)
        lens = (case["ctx"] + ql).to(dev).to(torch.int32)
        mx = int(lens.max())
        q = case["q"].permute(1, 0, 2, 3).contiguous()
        out = torch.empty((B, ql, case["H_q"], case["D"]), device=dev)
        st = max(args.split_tokens, 0)
        plan = pkv.multi_query_plan(B, ql, case["H_q"], case["k_cache"], mx, st,
                                    torch.cuda.get_device_properties(dev).multi_processor_count)
        ws = torch.empty(max(1, plan.workspace_bytes), dtype=torch.uint8, device=dev)
        fn = lambda: pkv.multi_query_attention(q, case["k_cache"], case["v_cache"], bt, lens, case["scale"], mx,
                                               split_tokens=st, out=out, workspace=ws)
        ms = _time_on_stream(fn, steps, warm, stream, sync)
        tr = _traced(pkv, fn, steps, sync)
        L = lens.double().cpu()
        kv = float(L.sum()) * case["H_kv"] * case["D"] * 4
        att = sum(float((L - ql + i + 1).clamp(min=0).sum()) for i in range(ql))
        flops = 4.0 * att * case["H_q"] * case["D"]
        n, t = tr.get("multi_query", (0, 0.0))
        k_ms = t / n if n else float("nan")
        achieved = kv / (k_ms / 1e3) / 1e9
        line.update({"metric": "multi-token query attention KV GB/s", "value": kv / ms / 1e6, "unit": "GB/s",
                     "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
                     "TFLOPs": flops / ms / 1e9,
                     "config": {"workload": args.workload, "q_len": ql, "B": B, "H_q": case["H_q"],
                                "H_kv": case["H_kv"], "d_head": case["D"], "block_size": case["bs"],
                                "split_tokens": plan.split_tokens, "splits": plan.max_splits,
                                "token_lanes": plan.workers},
                     "roofline": {"bound": "hbm", "kernel": "multi_query", "achieved": achieved, "peak": hbm,
                                  "unit": "GB/s", "frac": achieved / hbm,
                                  "peak_source": f"{hbm_kind} (hbm_gbs, copy bandwidth)",
                                  "algorithmic_bytes_per_launch": kv, "avg_launch_ms": k_ms,
                                  "tensor_TFLOPs": flops / (k_ms / 1e3) / 1e12, "traffic": None}})
        if not args.no_cpu_baseline:
            gbs, nu, procs, wall, ref = oracle_mq_throughput(case, q, lens, args.cpu_seconds)
            got = out.cpu().numpy()
            G = case["H_q"] // case["H_kv"]
            err = max(float(np.abs(got[b, :, h * G:(h + 1) * G] - r).max()) for (b, h), r in ref.items())
            line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": procs, "kind": "oracle",
                                    "sample": f"{nu} of {B * case['H_kv']} (sequence, KV head) units, "
                                              f"{wall:.1f} s wall, float64 numpy, one process per core"}
            line["parity"] = {"max_abs_err": err, "units": nu, "tolerance": 2e-3}
    else:
        nb, hkv, bs, d = 40000, 8, 16, 128
        kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
        blk = hkv * bs * d * 2
        g = torch.Generator().manual_seed(20260500)
        if args.op == "block_copy":
            npairs = 8192
            for c in (kc, vc):  # random bits, so that a copy shows
                c.view(torch.int16).copy_(torch.randint(-2**15, 2**15, c.shape, dtype=torch.int16, device=dev))
            perm = torch.randperm(nb, generator=g)
            src = perm[:npairs].to(torch.int32).to(dev)
            dst = perm[npairs:2 * npairs].to(torch.int32).to(dev)
            fn = lambda: pkv.copy_blocks(kc, vc, src, dst)
            ms = _time_on_stream(fn, steps, warm, stream, sync)
            byts = npairs * blk * 2 * 2
            gbs = byts / ms / 1e6
            line.update({"metric": "copy-on-write block copy GB/s (read + write)", "value": gbs, "unit": "GB/s",
                         "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
                         "config": {"pairs": npairs, "block_bytes_per_cache": blk, "pool_blocks": nb},
                         "roofline": {"bound": "hbm", "kernel": "block_copy", "achieved": gbs, "peak": hbm,
                                      "unit": "GB/s", "frac": gbs / hbm,
                                      "peak_source": f"{hbm_kind} (hbm_gbs, copy bandwidth)",
                                      "algorithmic_bytes_per_launch": byts, "avg_launch_ms": ms, "traffic": None}})
            if not args.no_cpu_baseline:
                # the oracle's copy on a sample of the pairs (host copies of
                # the blocks involved), timed, and the GPU pool checked against
                # it bit for bit
                from oracle.block_manager import copy_blocks as oracle_copy_blocks
                ns = 512
                s_ids, d_ids = src[:ns].cpu().tolist(), dst[:ns].cpu().tolist()
                sample = torch.tensor(s_ids + d_ids, dtype=torch.int64, device=dev)
                host = kc[sample].view(torch.int16).cpu().numpy()  # src blocks, then dst blocks
                pairs = [(i, ns + i) for i in range(ns)]
                t0 = time.perf_counter()
                want = oracle_copy_blocks(host, pairs)
                wall = time.perf_counter() - t0
                same = bool(np.array_equal(want[ns:], host[ns:]))   # the pool was copied already
                line["cpu_baseline"] = {"value": ns * blk * 2 / wall / 1e9, "unit": "GB/s", "cores": 1,
                                        "kind": "oracle", "sample": f"{ns} of {npairs} pairs of the K cache "
                                                                  f"(read + write), {wall * 1e3:.1f} ms, numpy"}
                line["parity"] = {"bit_exact": same, "pairs": ns}
        else:
            nh = 8192
            hk, hv = pkv.host_pool_like(kc, nh)
            src = torch.randperm(nb, generator=g)[:nh].to(torch.int32).to(dev)
            hdst = torch.randperm(nh, generator=g).to(torch.int32).to(dev)
            out_ms = _time_on_stream(lambda: pkv.copy_blocks_between(kc, vc, hk, hv, src, hdst), steps, warm,
                                     stream, sync)
            in_ms = _time_on_stream(lambda: pkv.copy_blocks_between(hk, hv, kc, vc, hdst, src), steps, warm,
                                    stream, sync)
            n = 2048
            ref_out = _time_on_stream(lambda: hk[:n].copy_(kc[:n], non_blocking=True), steps, warm, stream, sync)
            ref_in = _time_on_stream(lambda: kc[:n].copy_(hk[:n], non_blocking=True), steps, warm, stream, sync)
            byts = nh * blk * 2
            link_out = n * blk / ref_out / 1e6
            link_in = n * blk / ref_in / 1e6
            line.update({"metric": "host swap GB/s (device -> pinned host, host -> device)",
                         "value": byts / out_ms / 1e6, "unit": "GB/s", "stage_GBs": byts / in_ms / 1e6,
                         "ms_per_step": out_ms + in_ms, "higher_is_better": True, "dtype": "bf16",
                         "config": {"blocks": nh, "block_bytes_per_cache": blk},
                         "roofline": {"bound": "host link", "kernel": "block_copy",
                                      "achieved": byts / out_ms / 1e6, "peak": link_out, "unit": "GB/s",
                                      "frac": byts / out_ms / 1e6 / link_out,
                                      "peak_source": "one contiguous cudaMemcpyAsync of 64 MB each way, "
                                                     f"same run ({link_out:.0f} out, {link_in:.0f} in)",
                                      "traffic": None}})
    if pkv.device_error(dev) != 0:
        raise RuntimeError("device error")
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.op != "decode":
        run_op(args, int(os.environ.get("LOCAL_RANK", "0")))
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
