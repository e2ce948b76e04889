"""Seeded synthetic inputs shaped like the paged-decode workloads.

This module only draws random numbers and lays them out: context lengths,
shuffled physical block ids assigned to sequences, N(0,1) values for q / K / V,
and the FP8 scale rule of the FP8 workload (amax / 448 per sequence and KV
head).  It holds none of the method's arithmetic (no slot addressing, no
attention, no encoding), so the CUDA path and the CPU oracle can both be fed
from it.

Workloads (all 70B-class GQA except the tiny one: H_q = 64, H_kv = 8,
d_head = 128, the Llama-3-70B attention geometry used throughout the pages):

  tiny           B=2, context lengths {37, 100}, H_q=4, H_kv=1, D=64, block 16,
                 a pool of 32 blocks handed out in a seeded random order,
                 scale 1/8.
  gqa_bf16       B=64, context ~ U[512, 8192], block 16, bf16 KV, pool sized to
                 the blocks needed plus 10% free, shuffled.
  fp8            B=256, context ~ U[2048, 4096], block 16; K/V drawn in fp32
                 and written to an E4M3 cache by the append call with scale =
                 amax/448 per (sequence, KV head).
  shared_prefix  B=128, block 32; the first 4096 tokens of every sequence are
                 the same 128 physical blocks, then a private suffix of
                 U[64, 1024] tokens.
  long_ctx       B=8, context 131072, block 32, q drawn as 4 * N(0,1) (exact in
                 bf16), 32 decode steps with the context growing by one.

Every case covers ``steps`` decode steps: step s appends the token at logical
position ctx[b] + s of each sequence, then attends over ctx[b] + s + 1 tokens.
"""

import math

import torch

SPECS = {
    "tiny": dict(B=2, ctx=(37, 100), H_q=4, H_kv=1, D=64, bs=16, kv="bf16",
                 pool_blocks=32, scale=1.0 / 8.0, steps=1, seed=20260001),
    "gqa_bf16": dict(B=64, ctx_range=(512, 8192), H_q=64, H_kv=8, D=128, bs=16,
                     kv="bf16", free_frac=0.10, steps=1, seed=20260002),
    "fp8": dict(B=256, ctx_range=(2048, 4096), H_q=64, H_kv=8, D=128, bs=16,
                kv="e4m3", free_frac=0.10, steps=1, seed=20260003),
    "shared_prefix": dict(B=128, prefix=4096, suffix_range=(64, 1024), H_q=64, H_kv=8,
                          D=128, bs=32, kv="bf16", free_frac=0.10, steps=1, seed=20260004),
    "long_ctx": dict(B=8, ctx=(131072,) * 8, H_q=64, H_kv=8, D=128, bs=32, kv="bf16",
                     q_mult=4.0, free_frac=0.0, steps=32, seed=20260005),
}

WORKLOAD_ORDER = ["tiny", "gqa_bf16", "fp8", "shared_prefix", "long_ctx"]


def spec(name, **overrides):
    s = dict(SPECS[name])
    s.update(overrides)
    return s


def _ceil_div(a, b):
    return -(-a // b)


def draw_structure(s):
    """Context lengths, pool size and block tables (CPU, int tensors).

    Returns dict(ctx [B] int32 (before the first append), block_tables [B, MB]
    int32 with -1 past each sequence's blocks, num_blocks, shared_blocks).
    """
    g = torch.Generator().manual_seed(int(s["seed"]))
    B, bs, steps = s["B"], s["bs"], s.get("steps", 1)
    prefix = int(s.get("prefix", 0))
    if "ctx" in s:
        ctx = torch.tensor(list(s["ctx"]), dtype=torch.int64)
        assert ctx.numel() == B
    elif "ctx_range" in s:
        lo, hi = s["ctx_range"]
        ctx = torch.randint(lo, hi + 1, (B,), generator=g)
    else:
        lo, hi = s["suffix_range"]
        ctx = prefix + torch.randint(lo, hi + 1, (B,), generator=g)
    total = ctx + steps                                   # tokens after the last append
    need = [_ceil_div(int(t), bs) for t in total]
    shared = prefix // bs                                 # whole shared blocks
    private = [n - shared for n in need]
    used = shared + sum(private)
    if "pool_blocks" in s:
        nb = int(s["pool_blocks"])
    else:
        nb = int(math.ceil(used * (1.0 + s.get("free_frac", 0.0))))
    assert nb >= used
    perm = torch.randperm(nb, generator=g)
    mb = max(need)
    table = torch.full((B, mb), int(s.get("table_fill", -1)), dtype=torch.int64)
    cur = 0
    shared_ids = perm[cur:cur + shared]
    cur += shared
    for b in range(B):
        table[b, :shared] = shared_ids
        table[b, shared:need[b]] = perm[cur:cur + private[b]]
        cur += private[b]
    return dict(ctx=ctx.to(torch.int32), block_tables=table.to(torch.int32),
                num_blocks=nb, shared_blocks=shared, blocks_needed=need)


def make_case(name_or_spec, device="cpu", **overrides):
    """Draw one seeded case.

    Fields (torch tensors on ``device``):
      q             bf16 [steps, B, H_q, D]
      k_new, v_new  [steps, B, H_kv, D]      bf16 (bf16 cache) or fp32 (E4M3 cache)
      k_cache, v_cache  [NB, H_kv, bs, D]    bf16 filled with N(0,1) everywhere for
                                             bf16 caches; uint8 0x00 for E4M3
      block_tables  int32 [B, MB]            -1 past each sequence's blocks
      ctx           int32 [B]                tokens cached before the first append
    E4M3 cases add:
      fill_k, fill_v fp32 [N_fill, H_kv, D]  positions 0..ctx-1 of every sequence,
      fill_seq, fill_pos int64 [N_fill]      sequence-major
      k_scale, v_scale fp32 [B, H_kv]        amax / 448 over the sequence's
                                             ctx + steps tokens
    plus the scalars of the spec (B, H_q, H_kv, D, bs, kv, scale, steps).
    """
    s = spec(name_or_spec, **overrides) if isinstance(name_or_spec, str) else dict(name_or_spec, **overrides)
    st = draw_structure(s)
    B, H_q, H_kv, D, bs = s["B"], s["H_q"], s["H_kv"], s["D"], s["bs"]
    steps = s.get("steps", 1)
    nb = st["num_blocks"]
    dev = torch.device(device)
    gv = torch.Generator(device=dev).manual_seed(int(s["seed"]) * 7 + 1)
    case = dict(s)
    case.update(st)
    case.setdefault("scale", 1.0 / math.sqrt(D))
    case["steps"] = steps
    q = torch.randn((steps, B, H_q, D), generator=gv, device=dev) * float(s.get("q_mult", 1.0))
    case["q"] = q.to(torch.bfloat16)
    ctx = st["ctx"]
    if s["kv"] == "bf16":
        case["k_cache"] = torch.randn((nb, H_kv, bs, D), generator=gv, device=dev).to(torch.bfloat16)
        case["v_cache"] = torch.randn((nb, H_kv, bs, D), generator=gv, device=dev).to(torch.bfloat16)
        case["k_new"] = torch.randn((steps, B, H_kv, D), generator=gv, device=dev).to(torch.bfloat16)
        case["v_new"] = torch.randn((steps, B, H_kv, D), generator=gv, device=dev).to(torch.bfloat16)
    elif s["kv"] == "e4m3":
        case["k_cache"] = torch.zeros((nb, H_kv, bs, D), dtype=torch.uint8, device=dev)
        case["v_cache"] = torch.zeros((nb, H_kv, bs, D), dtype=torch.uint8, device=dev)
        n_fill = int(ctx.sum())
        case["fill_k"] = torch.randn((n_fill, H_kv, D), generator=gv, device=dev)
        case["fill_v"] = torch.randn((n_fill, H_kv, D), generator=gv, device=dev)
        case["fill_seq"] = torch.repeat_interleave(torch.arange(B), ctx.to(torch.int64))
        case["fill_pos"] = torch.cat([torch.arange(int(c)) for c in ctx]) if B else torch.zeros(0, dtype=torch.int64)
        case["k_new"] = torch.randn((steps, B, H_kv, D), generator=gv, device=dev)
        case["v_new"] = torch.randn((steps, B, H_kv, D), generator=gv, device=dev)
        # per (sequence, KV head) scale = amax / 448 over every token the
        # sequence will hold (the fill plus the appended tokens), in fp32
        seq_dev = case["fill_seq"].to(dev)
        for key, fill, new in (("k_scale", case["fill_k"], case["k_new"]),
                               ("v_scale", case["fill_v"], case["v_new"])):
            amax = torch.zeros((B, H_kv), dtype=torch.float32, device=dev)
            idx = seq_dev[:, None].expand(-1, H_kv)
            amax.scatter_reduce_(0, idx, fill.abs().amax(dim=2), "amax", include_self=True)
            amax = torch.maximum(amax, new.abs().amax(dim=3).amax(dim=0))
            case[key] = (amax / torch.tensor(448.0, dtype=torch.float32, device=dev)).contiguous()
    else:
        raise ValueError(s["kv"])
    return case
