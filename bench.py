"""Benchmark: paged decode attention KV GB/s and sequences/s on one GB300.

One step = one decode step of one attention layer for the whole batch:
pkv_decode_attention_append, all through the C ABI: every sequence's new
token is written into its slot (K/V scatter, bf16 copy or E4M3 quantisation)
by the decode launch itself, then the split-KV decode and the LSE combine.
(With --split-tokens -1, whose balanced mode has no fused append, the step
is pkv_append followed by pkv_decode_attention_ex.)

Default workload (the largest one-GPU configuration): long-context split-KV
decode, B=8 sequences of 131,072 tokens, H_q=64, H_kv=8, d_head=128, 32-token
blocks, bf16 KV, q drawn as 4*N(0,1); step s appends the token at position
131,072 + s and attends 131,073 + s tokens (about 4.3 GB of K/V read per
step, far larger than the 129 MB L2, so no flush is needed).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--repeats R]
                    [--impl ours|reference] [--workload NAME] [--no-workloads]

Prints one JSON line.  The K timed steps (steps 0..K-1, the context growing by
one token per step) are timed R times back to back, each repeat bracketed by
a barrier and a device synchronisation and replaying the same K steps from
the start (the appends rewrite the same slots with the same rows, so every
repeat does identical work); value = KV bytes attended over the K steps /
the median repeat's time (GB/s, 1e9 bytes), whole job over all ranks.  The
line's "workloads" key holds the same measurement for the other workloads
(tiny, gqa_bf16, fp8, shared_prefix), each with its oracle parity over every
(sequence, KV head) unit and the oracle's time beside it.

With --gpus N > 1 the script starts N ranks itself (torch.distributed.run on
127.0.0.1) unless it already runs under one: each rank runs an independent
replica on its own GPU (the path has no exchange step); value sums the ranks'
bytes over the slowest rank's time.  --dry-run replaces the GPU work by a host
loop (gloo), to check the launch and the reduction without a GPU.

--impl reference times the float64 CPU oracle (the reference of this
library) on the host cores over a bounded sample of the same workload.

--op cascade | multi_query | block_copy | host_swap times one of the other
hot-path operations instead of the decode step (one JSON line with "op").
"""

import argparse
import datetime
import hashlib
import json
import os
import socket
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
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal (~8 TB/s)
L2_BYTES = 129 * 1000 * 1000  # GB300 L2 (the flush writes twice this)
FALLBACK_BF16_TFLOPS = 1900.0
OTHER_WORKLOADS = ["tiny", "gqa_bf16", "fp8", "shared_prefix", "long_ctx"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--repeats", type=int, default=30,
                    help="times the K-step region is timed; value is the median")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None,
                    help="default: long_ctx (shared_prefix for --op cascade, gqa_bf16 for the other ops)")
    ap.add_argument("--op", default="decode",
                    choices=["decode", "cascade", "multi_query", "block_copy", "host_swap"],
                    help="decode (the headline step) or one of the other hot-path operations")
    ap.add_argument("--q-len", type=int, default=4, help="new tokens per sequence for --op multi_query")
    ap.add_argument("--split-tokens", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="decode: run the workload with its first BATCH sequences only (0: all); "
                         "for smaller profiler captures")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle (CPU baseline and parity)")
    ap.add_argument("--no-workloads", action="store_true", help="headline workload only")
    ap.add_argument("--dry-run", action="store_true", help="no GPU: check the rank launch and reduction")
    args = ap.parse_args(argv)
    if args.workload is None:
        args.workload = {"decode": "long_ctx", "cascade": "shared_prefix"}.get(args.op, "gqa_bf16")
    args.steps = max(1, args.steps)
    args.repeats = max(1, args.repeats)
    return args


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


def gather_ranks(x, device="cpu"):
    """[x of rank 0, x of rank 1, ...] (one element with one process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x)]
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    out = [torch.zeros_like(t) for _ in range(dist.get_world_size())]
    dist.all_gather(out, t)
    return [float(o.item()) for o in out]


def job_throughput(bytes_per_rank_step, steps, world, slowest_ms):
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return bytes_per_rank_step * steps * world / (slowest_ms / 1e3) / 1e9


def replica_seed(base_seed, rank):
    """Each replica draws its own workload (same shapes, different values)."""
    return base_seed + 1000 * rank


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return None


def measured_peaks():
    d = _peaks()
    if d and "hbm_gbs" in d:
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense bf16 tensor peak (burst: kernels timed on their own)."""
    d = _peaks()
    if d and "bf16_tflops" in d:
        return float(d["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("decode.cu", "decode_common.cuh", "pkv_device.cuh", "pkv_internal.h"):
        with open(os.path.join(ROOT, "paged_kv_cache_222_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, algo_bytes=None):
    """DRAM bytes per launch of the split kernel from a committed ncu summary,
    if it was taken on the current kernel source; else None.  A capture of a
    smaller batch of the same workload is scaled to `algo_bytes` by its ratio
    of DRAM bytes to algorithmic K/V bytes (traffic grows with the bytes
    attended)."""
    path = os.path.join(ROOT, "profiles", "decode_split_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    for r in rec.get("records", []):
        if r.get("workload") == workload and r.get("kernel_src") == kernel_source_hash():
            if r.get("dram_bytes_per_launch_full") is not None:
                return r["dram_bytes_per_launch_full"]
            if algo_bytes is not None and r.get("algorithmic_bytes"):
                return (r["dram_read"] + r["dram_write"]) / r["algorithmic_bytes"] * algo_bytes
    return None


def hbm_roofline(kernel, algo_bytes, avg_ms, workload=None):
    peak, kind = measured_peaks()
    achieved = algo_bytes / (avg_ms / 1e3) / 1e9 if avg_ms and avg_ms == avg_ms else None
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak if achieved else None,
            "frac_vs_nominal": achieved / NOMINAL_HBM_GBS if achieved else None,
            "peak_source": f"{kind} (hbm_gbs, copy bandwidth); frac_vs_nominal against 8000 GB/s",
            "kernel": kernel, "algorithmic_bytes_per_launch": algo_bytes, "avg_launch_ms": avg_ms,
            "traffic": recorded_traffic(workload, algo_bytes) if workload else None}


# ---------------------------------------------------------------- decode steps

class DecodeRun:
    """One workload set up on the device for K append + decode steps.

    Step i appends, for every sequence, the new token of generator step
    i % case_steps at position ctx + (i % case_steps) and decodes over the
    tokens up to it: the long-context workload's context grows by one token
    per step; the others (one step each) repeat their one step.  Slots come
    from the library's slot-mapping kernel, once for all steps, at set-up.
    """

    def __init__(self, name, steps, device, seed_offset=0, split_tokens=0, parity=True, batch=0):
        import torch
        import paged_kv_cache_222_gb300 as pkv
        import workloads as W
        from tests import oracle_pool as OP
        self.pkv, self.torch, self.dev = pkv, torch, device
        spec = W.spec(name)
        if 0 < batch < spec["B"]:
            spec["B"] = batch
            if "ctx" in spec:
                spec["ctx"] = tuple(spec["ctx"][:batch])
        grows = spec.get("steps", 1) > 1
        spec["steps"] = steps if grows else 1
        spec["seed"] = spec["seed"] + seed_offset
        self.name, self.grows = name, grows
        case = W.make_case(spec, device=device)
        self.case = case
        # generator inputs on the host, taken before the GPU touches the caches
        self.src = OP.UnitSource(case) if parity else None
        self.B, self.bs, self.S = case["B"], case["bs"], case["steps"]
        self.fp8 = case["kv"] == "e4m3"
        self.esz = 1 if self.fp8 else 2
        if self.fp8:
            from tests.gpu_support import fill_fp8_cache
            fill_fp8_cache(case)
        dev = device
        B, S = self.B, self.S
        self.bt = case["block_tables"].to(dev)
        ctx = case["ctx"].to(dev).to(torch.int64)
        ar = torch.arange(S, device=dev, dtype=torch.int64)
        pos = (ctx[None, :] + ar[:, None]).reshape(-1)                          # [S*B]
        seq = torch.arange(B, device=dev, dtype=torch.int64).repeat(S)
        self.slots = pkv.slot_mapping(self.bt, pos, case["k_cache"], seq_index=seq).view(S, B)
        self.lens = (ctx[None, :] + ar[:, None] + 1).to(torch.int32).contiguous()   # [S, B]
        self.max_len = int(case["ctx"].max()) + S                                   # bound for every step
        self.q = case["q"].contiguous()
        self.kn = case["k_new"].contiguous()
        self.vn = case["v_new"].contiguous()
        self.ks = case.get("k_scale") if self.fp8 else None
        self.vs = case.get("v_scale") if self.fp8 else None
        self.out = torch.empty((B, case["H_q"], case["D"]), dtype=torch.float32, device=dev)
        self.split_tokens = split_tokens
        self.plan = pkv.decode_plan(B, case["H_q"], case["k_cache"], self.max_len, split_tokens,
                                    torch.cuda.get_device_properties(dev).multi_processor_count)
        self.ws = torch.empty(max(1, int(self.plan.workspace_bytes)), dtype=torch.uint8, device=dev)
        ctx_h = case["ctx"].to(torch.float64)
        per_tok = case["H_kv"] * case["D"] * 2 * self.esz
        self.step_bytes = [float((ctx_h + s + 1).sum()) * per_tok for s in range(S)]
        self.per_tok = per_tok
        torch.cuda.synchronize(dev)

    def step_index(self, i):
        return i % self.S

    @property
    def fused(self):
        """The step appends inside the decode launch (every mode but the
        balanced one)."""
        return self.split_tokens >= 0

    def step(self, i, q=None, kn=None, vn=None, slots=None, bt=None, lens=None, out=None):
        s = self.step_index(i)
        c = self.case
        kn = self.kn[s] if kn is None else kn
        vn = self.vn[s] if vn is None else vn
        extra = {}
        if self.fused:
            extra = dict(k_new=kn, v_new=vn)
        else:
            self.pkv.append(kn, vn, self.slots[s] if slots is None else slots, c["k_cache"], c["v_cache"],
                            self.ks, self.vs)
        self.pkv.decode_attention(self.q[s] if q is None else q, c["k_cache"], c["v_cache"],
                                  self.bt if bt is None else bt, self.lens[s] if lens is None else lens,
                                  c["scale"], self.ks, self.vs, max_context_len=self.max_len,
                                  out=self.out if out is None else out, split_tokens=self.split_tokens,
                                  workspace=self.ws, **extra)

    def region_bytes(self, k):
        return sum(self.step_bytes[self.step_index(i)] for i in range(k))

    def config(self):
        c = self.case
        ctx = c["ctx"]
        p = self.plan
        cfg = {"workload": self.name, "B": self.B, "H_q": c["H_q"], "H_kv": c["H_kv"], "d_head": c["D"],
               "block_size": self.bs, "kv_dtype": c["kv"],
               "context_attended": f"{int(ctx.min()) + 1}..{int(ctx.max()) + self.S} "
                                   f"(mean {float(ctx.float().mean()) + 1:.0f} at the first step)",
               "context_growth": "one token per step" if self.grows else "the same step repeated",
               "kv_bytes_per_step": sum(self.step_bytes) / self.S,
               "split": ("balanced ranges over %d warps" % p.workers) if p.mode == 0
                        else ("%d tokens x %d splits" % (p.split_tokens, p.max_splits)),
               "l2": "inputs larger than L2 (no flush)" if self.step_bytes[0] > L2_BYTES else
                     "L2 flushed between steps (258 MB write outside each step's events)",
               "append": "fused into the decode launch" if self.fused else "a launch of its own",
               "parallelism": "replicas"}
        if c.get("prefix", 0):
            cfg["shared_prefix_tokens"] = int(c["prefix"])
        return cfg

    def oracle_parity(self, seconds=None):
        """The last step's output (held in self.out after a region) against
        the oracle on every (sequence, KV head) unit (or as many as `seconds`
        allows).  Returns (parity dict, cpu_baseline dict)."""
        from tests import oracle_pool as OP
        c = self.case
        last = self.S - 1
        units = [(b, h) for b in range(self.B) for h in range(c["H_kv"])]
        got = self.out.cpu().numpy()
        res = OP.run_units(self.src, units, last + 1, [last], seconds=seconds)
        G = c["H_q"] // c["H_kv"]
        err = OP.max_abs_err(got, res["outputs"], G)
        tol = 5e-3 if self.fp8 else 2e-3
        parity = {"max_abs_err": err, "units": res["units"], "of_units": len(units), "step": last,
                  "tolerance": tol, "ok": bool(err <= tol)}
        cpu = {"value": res["kv_bytes"] / res["wall"] / 1e9, "unit": "GB/s", "cores": res["procs"],
               "kind": "oracle",
               "sample": f"{res['units']} of {len(units)} (sequence, KV head) units of step {last} of the "
                         f"{self.name} workload (the oracle appends steps 0..{last} itself), "
                         f"{res['wall']:.1f} s wall, float64 numpy, one process per core",
               "oracle_s_per_step": res["wall"] * len(units) / max(1, res["units"])}
        return parity, cpu

    def free(self):
        for k in ("case", "src", "slots", "lens", "q", "kn", "vn", "out", "ws", "bt"):
            setattr(self, k, None)


def _barrier(dist, dev):
    import torch
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)


def time_regions(run, k, repeats, dist, dev, scrub=None):
    """Time the K-step region `repeats` times; returns the ms of each repeat
    (the slowest rank's).  With `scrub` (an L2-sized buffer) every step is
    timed on its own with the buffer written between steps, outside the
    events."""
    import torch
    stream = torch.cuda.current_stream(dev)
    out = []
    for _ in range(repeats):
        _barrier(dist, dev)
        if scrub is not None:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(k)]
            for i, (a, b) in enumerate(evs):
                scrub.zero_()
                a.record(stream)
                run.step(i)
                b.record(stream)
        else:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(k):
                run.step(i)
            e1.record(stream)
        _barrier(dist, dev)
        ms = sum(a.elapsed_time(b) for a, b in evs) if scrub is not None else e0.elapsed_time(e1)
        out.append(max_over_ranks(ms, dev))
    return out


def traced_region(run, k, dev):
    """One more region with every library launch bracketed by CUDA events on
    its own stream: {kernel: (launches, total ms)} (event records sit between
    the kernels, so this pass is not the one `value` comes from)."""
    import torch
    pkv = run.pkv
    pkv.trace_read()
    pkv.trace_enable(True)
    for i in range(k):
        run.step(i)
    torch.cuda.synchronize(dev)
    pkv.trace_enable(False)
    return pkv.trace_read()


def e2e_region(run, k, repeats, dist, dev, world):
    """The same K steps end to end through the public API with host buffers:
    every step copies its inputs (q, the new K/V rows, block tables, lengths;
    the slots too when the append is a launch of its own) from pinned host
    memory and reads its output back, on a copy
    stream one step ahead of the compute (two sets of device buffers); the
    timed region spans every copy.  Returns (GB/s of the median repeat,
    h2d bytes per step, d2h bytes per step)."""
    import torch
    stream = torch.cuda.current_stream(dev)
    pin = lambda t: t.cpu().pin_memory()
    S = run.S
    h_in = [[pin(run.q[s]), pin(run.kn[s]), pin(run.vn[s]), pin(run.bt), pin(run.lens[s])]
            + ([] if run.fused else [pin(run.slots[s])]) for s in range(S)]
    h_outs = [torch.empty(run.out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    d_in = [[torch.empty_like(t, device=dev) for t in h_in[0]] for _ in range(2)]
    d_out = [torch.empty_like(run.out) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in[0])
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    cstream = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]

    def h2d_copy(i):  # on the copy stream
        if i >= 2:
            cstream.wait_event(ev_done[i % 2])     # step i-2 is done with this set
        for d, h in zip(d_in[i % 2], h_in[run.step_index(i)]):
            d.copy_(h, non_blocking=True)
        ev_in[i % 2].record(cstream)

    def one(n):
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
            q, kn, vn, bt, ln = d_in[i % 2][:5]
            sl = None if run.fused else d_in[i % 2][5]
            run.step(i, q=q, kn=kn, vn=vn, slots=sl, bt=bt, lens=ln, out=d_out[i % 2])
            ev_done[i % 2].record(stream)
            with torch.cuda.stream(cstream):
                cstream.wait_event(ev_done[i % 2])
                h_outs[i % 2].copy_(d_out[i % 2], non_blocking=True)
        tail = torch.cuda.Event()
        tail.record(cstream)
        stream.wait_event(tail)
        end.record(stream)
        return start, end

    one(min(3, k))
    vals = []
    for _ in range(repeats):
        _barrier(dist, dev)
        e0, e1 = one(k)
        _barrier(dist, dev)
        vals.append(job_throughput(run.region_bytes(k), 1, world, max_over_ranks(e0.elapsed_time(e1), dev)))
    return statistics.median(vals), h2d, d2h


def measure_workload(run, args, dist, dev, world, rank, with_e2e):
    """Warm-up, R timed repeats of K steps, a traced pass, optionally e2e, and
    the oracle.  Returns the measurement as a dict (rank 0's view)."""
    import torch
    pkv = run.pkv
    k = args.steps
    for i in range(max(3, args.warmup)):
        run.step(i)
    torch.cuda.synchronize(dev)
    if pkv.device_error(dev) != 0:
        raise RuntimeError(f"{run.name}: device error during warm-up")
    flush = run.step_bytes[0] <= L2_BYTES
    scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    t0 = time.time()
    reps = time_regions(run, k, args.repeats, dist, dev, scrub)
    t1 = time.time()
    clocks.stop()
    clk = clocks.summary(t0, t1)
    del scrub
    trace = traced_region(run, k, dev)
    region = run.region_bytes(k)
    gbs = [job_throughput(region, 1, world, ms) for ms in reps]
    med_ms = statistics.median(reps)
    split = trace.get("decode_split", (0, 0.0))
    avg_ms = split[1] / split[0] if split[0] else float("nan")
    launches = sum(n for n, _ in trace.values())
    res = {
        "value": job_throughput(region, 1, world, med_ms), "unit": "GB/s",
        "ms_per_step": med_ms / k, "seqs_per_s": run.B * k * world / (med_ms / 1e3),
        "steps": k, "repeats": args.repeats,
        "spread_GBs": {"min": min(gbs), "median": statistics.median(gbs), "max": max(gbs)},
        "config": run.config(),
        "roofline": hbm_roofline("decode_split", region / k, avg_ms, run.name),
        "kernel_times_ms": {kk: {"launches": n, "avg_ms": t / n} for kk, (n, t) in trace.items() if n},
        "gpu_launches": launches * args.repeats, "gpu_launches_per_step": launches / k,
        "clocks": clk,
    }
    if flush:
        res["us_per_step"] = med_ms / k * 1e3
    if run.case.get("prefix", 0):
        res["roofline"]["note"] = ("logical bytes: every sequence reads the shared prefix blocks, which stay in "
                                   "L2 after the first reader, so the fraction exceeds 1; see unique_GBs")
        c = run.case
        pre = int(c["prefix"])
        uniq = sum((pre + float((c["ctx"].double() + run.step_index(i) + 1 - pre).sum())) * run.per_tok
                   for i in range(k))
        res["unique_GBs"] = res["value"] * uniq / region
    if with_e2e:
        e2e, h2d, d2h = e2e_region(run, k, args.repeats, dist, dev, world)
        res["e2e"] = {"value": e2e, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "steps": k, "repeats": args.repeats}
    if pkv.device_error(dev) != 0:
        raise RuntimeError(f"{run.name}: device error during the timed region")
    if run.src is not None and rank == 0:
        # `run.out` holds the last step's output (the traced pass ends on it)
        parity, cpu = run.oracle_parity()
        res["parity"] = parity
        res["cpu_baseline"] = cpu
    return res


def cascade_on(run, args, dev):
    """The cascade call on a shared-prefix workload (after its decode
    measurement): ms per call (median of R repeats of K calls), logical and
    unique KV GB/s, and its max-abs difference from the plain decode."""
    import torch
    pkv, c = run.pkv, run.case
    s = run.S - 1
    pre = int(c["prefix"])
    pblocks = run.bt[0, :pre // run.bs].contiguous()
    plan = pkv.cascade_plan(run.B, c["H_q"], c["k_cache"], pre, run.max_len,
                            torch.cuda.get_device_properties(dev).multi_processor_count)
    ws = torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=dev)
    out = torch.empty_like(run.out)
    fn = lambda: pkv.cascade_decode_attention(run.q[s], c["k_cache"], c["v_cache"], pblocks, pre, run.bt,
                                              run.lens[s], c["scale"], run.max_len, out=out, workspace=ws)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        fn()
    reps = []
    for _ in range(args.repeats):
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        reps.append(e0.elapsed_time(e1) / args.steps)
    ms = statistics.median(reps)
    logical = run.step_bytes[s]
    unique = (pre + float((c["ctx"].double() + s + 1 - pre).sum())) * run.per_tok
    return {"ms_per_call": ms, "logical_GBs": logical / ms / 1e6, "unique_GBs": unique / ms / 1e6,
            "max_abs_diff_vs_plain_decode": float((out - run.out).abs().max())}


# ---------------------------------------------------------------- arms

def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is a bounded sample of
    the workload's (sequence, KV head) units (the oracle appends the step's
    tokens itself)."""
    if rank != 0:
        return
    import numpy as np
    import workloads as W
    from tests import oracle_pool as OP
    spec = W.spec(args.workload)
    grows = spec.get("steps", 1) > 1
    spec["steps"] = args.steps if grows else 1
    case = W.make_case(spec, device="cpu")
    src = OP.UnitSource(case)
    n_steps = spec["steps"]
    per_step = max(2.0, min(8.0, 120.0 / max(1, args.steps + args.warmup)))
    units = [(b, h) for b in range(case["B"]) for h in range(case["H_kv"])]
    vals, cores, done = [], None, 0
    for i in range(args.warmup + args.steps):
        s = i % n_steps
        order = list(units)
        np.random.default_rng(i).shuffle(order)
        res = OP.run_units(src, order, s + 1, [s], seconds=per_step)
        cores = res["procs"]
        if i >= args.warmup:
            vals.append(res["kv_bytes"] / res["wall"] / 1e9)
            done += res["units"]
    value = statistics.median(vals) if vals else 0.0
    esz = 1 if case["kv"] == "e4m3" else 2
    kv_bytes = float((case["ctx"].double() + 1).sum()) * case["H_kv"] * case["D"] * 2 * esz
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": kv_bytes / (value * 1e9) * 1e3 if value else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.workload, "B": case["B"], "H_q": case["H_q"], "H_kv": case["H_kv"],
                       "d_head": case["D"], "block_size": case["bs"], "kv_bytes_per_step": kv_bytes},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{done} (sequence, KV head) units over {args.steps} steps of "
                                       f"~{per_step:.0f} s each; float64 numpy oracle, one process per core"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    from paged_kv_cache_222_gb300 import build

    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
    cpu = not args.no_cpu_baseline and world == 1
    run = DecodeRun(args.workload, args.steps, dev, seed_offset=replica_seed(0, rank),
                    split_tokens=args.split_tokens, parity=cpu, batch=args.batch)
    m = measure_workload(run, args, dist, dev, world, rank, with_e2e=True)
    dtype = "e4m3" if run.fp8 else "bf16"
    cascade = cascade_on(run, args, dev) if run.case.get("prefix", 0) else None
    run.free()
    del run
    torch.cuda.empty_cache()

    others = {}
    if world == 1 and not args.no_workloads:
        for name in OTHER_WORKLOADS:
            if name == args.workload:
                continue
            r = DecodeRun(name, args.steps, dev, split_tokens=args.split_tokens, parity=cpu)
            w = measure_workload(r, args, None, dev, 1, rank, with_e2e=False)
            if r.case.get("prefix", 0):
                w["cascade"] = cascade_on(r, args, dev)
            w["dtype"] = "e4m3" if r.fp8 else "bf16"
            w.pop("clocks", None)
            others[name] = w
            r.free()
            del r
            torch.cuda.empty_cache()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": m["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "repeats": args.repeats, "ms_per_step": m["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic",
        "config": m["config"], "seqs_per_s": m["seqs_per_s"], "spread_GBs": m["spread_GBs"],
        "roofline": m["roofline"], "kernel_times_ms": m["kernel_times_ms"], "e2e": m["e2e"],
        "clocks": m["clocks"], "gpu_launches": m["gpu_launches"],
        "gpu_launches_per_step": m["gpu_launches_per_step"],
    }
    for key in ("unique_GBs", "us_per_step", "parity", "cpu_baseline"):
        if key in m:
            line[key] = m[key]
    if cascade is not None:
        line["cascade"] = cascade
    if others:
        line["workloads"] = others
    print(json.dumps(line), flush=True)


def run_dry(args, rank, world):
    """No GPU: each rank times a host loop as its 'steps'; the same barrier,
    max-over-ranks and whole-job arithmetic as the GPU path (gloo)."""
    import numpy as np
    dist = None
    if world > 1:
        import torch.distributed as dist
    a = np.random.default_rng(rank).standard_normal(1 << 16)
    for _ in range(args.warmup):
        float(a.sum())
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        float((a * a).sum())
    ms = (time.perf_counter() - t0) * 1e3
    if dist is not None:
        dist.barrier()
    slowest = max_over_ranks(ms)
    per_rank = gather_ranks(ms)
    if rank == 0:
        nbytes = a.nbytes
        print(json.dumps({"metric": "dry run (host loop; no GPU)", "value": job_throughput(nbytes, args.steps, world,
                                                                                           max(slowest, 1e-6)),
                          "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ranks_reported": len(per_rank), "rank_ms": per_rank, "slowest_ms": slowest,
                          "dry_run": True}), flush=True)


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


def _append_steps(pkv, case, n, dev):
    """Append the first n generator steps' tokens of every sequence."""
    import torch
    bt = case["block_tables"].to(dev)
    ctx = case["ctx"].to(dev).to(torch.int64)
    for s in range(n):
        slots = pkv.slot_mapping(bt, ctx + s, case["k_cache"])
        pkv.append(case["k_new"][s].contiguous(), case["v_new"][s].contiguous(), slots,
                   case["k_cache"], case["v_cache"])


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
    from tests import oracle_pool as OP

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
        src = None if args.no_cpu_baseline else OP.UnitSource(case)
        _append_steps(pkv, case, 1, dev)
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
        ms_plain = _time_on_stream(plain, steps, warm, stream, sync)
        ms = _time_on_stream(fn, steps, warm, stream, sync)
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
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        row_blocks = -(-B * (case["H_q"] // case["H_kv"]) // 256) * case["H_kv"]
        sm_share = min(1.0, row_blocks * plan.workers / sms)   # SMs the prefix CTAs hold (one per SM)
        prefix_line = {"bound": "tensor", "kernel": "cascade_prefix", "achieved": achieved, "peak": tf_peak,
                       "unit": "TFLOP/s", "frac": achieved / tf_peak,
                       "peak_source": f"{tf_kind} (bf16_tflops, burst)", "algorithmic_flops_per_launch": flops,
                       "avg_launch_ms": pf_ms, "sm_share": sm_share,
                       "frac_of_its_sms": achieved / (tf_peak * sm_share), "traffic": None}
        suffix_line = hbm_roofline("decode_split (suffixes, beside the prefix)", suffix_bytes, sf_ms)
        # the roofline line is the kernel that holds more SM time (its duration
        # times the SMs it runs on: the prefix CTAs hold sm_share of them, the
        # suffix decode the rest); the other rides along
        pf_smt, sf_smt = pf_ms * sm_share, sf_ms * (1.0 - sm_share)
        dominant, other = (prefix_line, suffix_line) if pf_smt > sf_smt else (suffix_line, prefix_line)
        floor_ms = unique / (hbm * 1e9) * 1e3
        line.update({"metric": "cascade decode KV GB/s (logical bytes: every sequence's whole context)",
                     "value": logical / ms / 1e6, "unit": "GB/s", "ms_per_step": ms, "higher_is_better": True,
                     "dtype": "bf16", "unique_GBs": unique / ms / 1e6, "plain_decode_ms": ms_plain,
                     "unique_bytes_floor_ms": floor_ms, "frac_of_unique_floor": floor_ms / ms,
                     "config": {"workload": args.workload, "B": B, "H_q": case["H_q"], "H_kv": case["H_kv"],
                                "d_head": case["D"], "block_size": bs, "shared_prefix": prefix,
                                "prefix_ranges": plan.workers, "prefix_range_tokens": plan.prefix_split_tokens,
                                "suffix_split_tokens": plan.split_tokens},
                     "kernel_times_ms": {k: {"launches": nn, "avg_ms": tt / nn} for k, (nn, tt) in tr.items() if nn},
                     "roofline": dominant, "roofline_other_kernel": other})
        if src is not None:
            # the oracle (plain decode of every sequence's whole context; the
            # cascade reaches the same result) on every (sequence, KV head) unit
            units = [(b, h) for b in range(B) for h in range(case["H_kv"])]
            res = OP.run_units(src, units, 1, [0])
            err = OP.max_abs_err(out.cpu().numpy(), res["outputs"], case["H_q"] // case["H_kv"])
            line["cpu_baseline"] = {"value": res["kv_bytes"] / res["wall"] / 1e9, "unit": "GB/s",
                                    "cores": res["procs"], "kind": "oracle",
                                    "sample": f"{res['units']} of {len(units)} (sequence, KV head) units, "
                                              f"{res['wall']:.1f} s wall, float64 numpy, one process per core"}
            line["parity"] = {"max_abs_err": err, "units": res["units"], "tolerance": 2e-3}
    elif args.op == "multi_query":
        ql = args.q_len
        case = W.make_case(args.workload, device=dev, steps=ql)
        src = None if args.no_cpu_baseline else OP.UnitSource(case)
        _append_steps(pkv, case, ql, dev)
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
        roof = hbm_roofline("multi_query", kv, k_ms)
        roof["tensor_TFLOPs"] = flops / (k_ms / 1e3) / 1e12
        line.update({"metric": "multi-token query attention KV GB/s", "value": kv / ms / 1e6, "unit": "GB/s",
                     "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
                     "TFLOPs": flops / ms / 1e9,
                     "config": {"workload": args.workload, "q_len": ql, "B": B, "H_q": case["H_q"],
                                "H_kv": case["H_kv"], "d_head": case["D"], "block_size": case["bs"],
                                "split_tokens": plan.split_tokens, "splits": plan.max_splits,
                                "token_lanes": plan.workers},
                     "roofline": roof})
        if src is not None:
            units = [(b, h) for b in range(B) for h in range(case["H_kv"])]
            res = OP.run_units(src, units, ql, list(range(ql)))
            err = OP.max_abs_err(out.cpu().numpy(), res["outputs"], case["H_q"] // case["H_kv"], multi=True)
            line["cpu_baseline"] = {"value": res["kv_bytes"] / res["wall"] / 1e9, "unit": "GB/s",
                                    "cores": res["procs"], "kind": "oracle",
                                    "sample": f"{res['units']} of {len(units)} (sequence, KV head) units, "
                                              f"{res['wall']:.1f} s wall, float64 numpy, one process per core"}
            line["parity"] = {"max_abs_err": err, "units": res["units"], "tolerance": 2e-3}
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
            roof = hbm_roofline("block_copy", byts, ms)
            line.update({"metric": "copy-on-write block copy GB/s (read + write)", "value": gbs, "unit": "GB/s",
                         "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
                         "config": {"pairs": npairs, "block_bytes_per_cache": blk, "pool_blocks": nb},
                         "roofline": roof})
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


# ---------------------------------------------------------------- launch

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_replicas(args, argv):
    """Start args.gpus ranks of this script under torch.distributed.run (one
    per GPU, rendezvous on 127.0.0.1) and return its exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_replicas(args, argv))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.dry_run:
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        try:
            run_dry(args, rank, world)
        finally:
            if world > 1:
                import torch.distributed as dist
                dist.destroy_process_group()
        return
    if args.op != "decode":
        if rank == 0:
            run_op(args, local_rank)
        return
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
