"""Oracle references for many (sequence, KV head) units at once.

Harness code for the GPU tests and bench.py: it feeds the float64 oracle
(``oracle.paged_attention``) and runs it in a spawn pool of one
single-threaded process per host core.

Every input comes from the workload generator, never from the CUDA path: a
host copy of the caches taken before any append (bf16 caches, as drawn), the
FP8 fill rows and scales (the oracle writes an E4M3 cache itself with its own
append), the new tokens' rows and the queries.  A worker rebuilds one unit's
cache (the sequence's blocks renumbered 0..n-1, one KV head, which leaves the
result unchanged), applies the appends of the steps up to the one asked for
with the oracle's append, and runs the oracle's decode (or multi-token
attention).
"""

import collections
import os
import time

import numpy as np
import torch

_E4M3_NAN = 0x7F


def _bits16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


class UnitSource:
    """Host copies of a workload case's generator inputs, taken before any
    append into its caches."""

    def __init__(self, case):
        self.B, self.H_q, self.H_kv, self.D = case["B"], case["H_q"], case["H_kv"], case["D"]
        self.G = self.H_q // self.H_kv
        self.bs, self.kv, self.scale = case["bs"], case["kv"], float(case["scale"])
        self.ctx = case["ctx"].cpu().to(torch.int64).numpy()
        self.need = list(case["blocks_needed"])
        self.tables = case["block_tables"].cpu()
        self.q = case["q"].cpu()                                  # [steps, B, H_q, D] bf16
        if self.kv == "bf16":
            # head-major copies [H_kv, num_blocks, bs, D]: one head's blocks
            # gather as contiguous rows
            self.k_cache = case["k_cache"].cpu().transpose(0, 1).contiguous()
            self.v_cache = case["v_cache"].cpu().transpose(0, 1).contiguous()
            self.k_new = case["k_new"].cpu()
            self.v_new = case["v_new"].cpu()
        else:
            self.fill_k = case["fill_k"].cpu()
            self.fill_v = case["fill_v"].cpu()
            self.fill_start = np.concatenate([[0], np.cumsum(self.ctx)])
            self.k_scale = case["k_scale"].cpu().numpy()
            self.v_scale = case["v_scale"].cpu().numpy()
            self.k_new = case["k_new"].cpu()
            self.v_new = case["v_new"].cpu()

    def kv_bytes(self, b, n_new):
        """K and V bytes of one unit attended after n_new appends."""
        p = 2 if self.kv == "bf16" else 1
        return (int(self.ctx[b]) + n_new) * self.D * 2 * p

    def payload(self, b, h, n_new, q_steps):
        """Inputs of unit (b, h) with the first n_new new tokens appended and
        queries q[q_steps] (one step for decode, several for multi-token)."""
        n = self.need[b]
        g = slice(h * self.G, (h + 1) * self.G)
        q = _bits16(self.q[q_steps, b, g])                      # [len(q_steps), G, D]
        if self.kv == "bf16":
            ids = self.tables[b, :n].to(torch.int64)
            # only head h of the sequence's blocks: [n, 1, bs, D]
            kb = torch.index_select(self.k_cache[h], 0, ids).unsqueeze(1)
            vb = torch.index_select(self.v_cache[h], 0, ids).unsqueeze(1)
            raw = dict(k=_bits16(kb), v=_bits16(vb),
                       k_new=_bits16(self.k_new[:n_new, b, h:h + 1]),
                       v_new=_bits16(self.v_new[:n_new, b, h:h + 1]))
        else:
            a, e = int(self.fill_start[b]), int(self.fill_start[b + 1])
            raw = dict(fill_k=self.fill_k[a:e, h:h + 1].numpy(), fill_v=self.fill_v[a:e, h:h + 1].numpy(),
                       k_new=self.k_new[:n_new, b, h:h + 1].numpy(), v_new=self.v_new[:n_new, b, h:h + 1].numpy(),
                       ks=np.float32(self.k_scale[b, h]), vs=np.float32(self.v_scale[b, h]))
        return dict(key=(b, h), kv=self.kv, n=n, bs=self.bs, D=self.D, ctx=int(self.ctx[b]), n_new=n_new,
                    q=q, scale=self.scale, **raw)


def unit_worker(p):
    """Oracle output of one unit: decode ([G, D]) when one query step is
    given, else multi-token attention ([q_len, G, D]); with E4M3 caches also
    the codes of every position written ([tokens, D] for K and V)."""
    from oracle import paged_attention as PA
    t0 = time.perf_counter()
    n, bs, D, ctx, n_new = p["n"], p["bs"], p["D"], p["ctx"], p["n_new"]
    table = np.arange(n, dtype=np.int32)[None, :]
    new_slots = np.array([PA.slot_of(table[0], ctx + s, bs) for s in range(n_new)], dtype=np.int64)
    if p["kv"] == "bf16":
        dt, src, ks, vs = PA.BF16, PA.BF16, None, None
        kc, vc = p["k"], p["v"]
    else:
        dt, src = PA.E4M3, PA.F32
        ks = np.array([p["ks"]], dtype=np.float32)
        vs = np.array([p["vs"]], dtype=np.float32)
        kc = np.full((n, 1, bs, D), _E4M3_NAN, dtype=np.uint8)
        vc = kc.copy()
        fill_slots = np.array([PA.slot_of(table[0], t, bs) for t in range(ctx)], dtype=np.int64)
        kc, vc = PA.append(p["fill_k"], p["fill_v"], src, fill_slots, kc, vc, dt, ks, vs, scale_row_stride=0)
    if n_new:
        kc, vc = PA.append(p["k_new"], p["v_new"], src, new_slots, kc, vc, dt, ks, vs, scale_row_stride=0)
    total = ctx + n_new
    ksc = None if ks is None else ks[None, :]
    vsc = None if vs is None else vs[None, :]
    q = p["q"]
    if q.shape[0] == 1:
        out = PA.decode_attention(q, kc, vc, dt, table, np.array([total]), p["scale"], ksc, vsc)[0]
    else:
        out = PA.multi_query_attention(q[None], kc, vc, dt, table, np.array([total]), p["scale"], ksc, vsc)[0]
    codes = None
    if p["kv"] != "bf16":
        codes = (kc[:, 0].reshape(n * bs, D)[:total].copy(), vc[:, 0].reshape(n * bs, D)[:total].copy())
    return time.perf_counter() - t0, p["key"], out, codes


def _warm(_):
    import numpy  # noqa: F401
    from oracle import paged_attention  # noqa: F401
    return 0


def host_procs():
    return max(1, min(len(os.sched_getaffinity(0)), 32))


def run_units(src, units, n_new, q_steps, seconds=None, want_codes=False, procs=None):
    """Oracle outputs of `units` [(b, h)] after n_new appends, queries
    q[q_steps]; in a spawn pool of `procs` single-threaded processes (one per
    host core by default), at most two units per process in flight.  With
    `seconds`, no unit is started after that much wall time.

    Returns dict(outputs={(b, h): out}, codes={(b, h): (k, v)} (E4M3 only),
    units=done, procs, wall=seconds, kv_bytes=K and V bytes attended)."""
    import multiprocessing as mp
    procs = procs or host_procs()
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    outputs, codes = {}, {}
    kv_bytes = 0
    with mp.get_context("spawn").Pool(procs) as pool:
        pool.map(_warm, range(procs))
        t0 = time.perf_counter()
        it = iter(units)
        pending = collections.deque()
        while True:
            while len(pending) < 2 * procs and (seconds is None or time.perf_counter() - t0 < seconds):
                u = next(it, None)
                if u is None:
                    break
                pending.append(pool.apply_async(unit_worker, (src.payload(u[0], u[1], n_new, q_steps),)))
            if not pending:
                break
            _, key, out, cd = pending.popleft().get()
            outputs[key] = out
            if want_codes and cd is not None:
                codes[key] = cd
            kv_bytes += src.kv_bytes(key[0], n_new)
        wall = time.perf_counter() - t0
    return dict(outputs=outputs, codes=codes, units=len(outputs), procs=procs, wall=wall, kv_bytes=kv_bytes)


def max_abs_err(got, outputs, G, multi=False):
    """Largest |GPU - oracle| over the units in `outputs`; got is the GPU
    output as numpy ([B, H_q, D], or [B, q_len, H_q, D] when multi)."""
    worst = 0.0
    for (b, h), ref in outputs.items():
        g = got[b, :, h * G:(h + 1) * G] if multi else got[b, h * G:(h + 1) * G]
        worst = max(worst, float(np.max(np.abs(g - ref))))
    return worst
