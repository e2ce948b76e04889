"""Helpers shared by the GPU parity tests: run decode steps through the C ABI,
and compute oracle references for chosen (sequence, KV head) units from the
generator's inputs only (never from anything the CUDA path wrote)."""

import numpy as np
import torch

import paged_kv_cache_222_gb300 as pkv
from oracle import formats as F
from oracle import paged_attention as PA

BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F


def bits16(t):
    """Raw uint16 words of a bf16 tensor (any device) as numpy."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bytes8(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def poison_unused(case):
    """Fill every slot no sequence will hold (free blocks, and the tail of each
    sequence's last block) with NaN, in place, on the case's device."""
    kc, vc = case["k_cache"], case["v_cache"]
    bs = case["bs"]
    nan = BF16_NAN if case["kv"] == "bf16" else E4M3_NAN
    used = np.zeros(case["num_blocks"], dtype=bool)
    bt = case["block_tables"].cpu().numpy()
    slots = []
    for b in range(case["B"]):
        n = case["blocks_needed"][b]
        used[bt[b, :n]] = True
        for pos in range(int(case["ctx"][b]) + case["steps"], n * bs):
            slots.append(PA.slot_of(bt[b], pos, bs))
    free = torch.from_numpy(np.nonzero(~used)[0]).to(kc.device)
    view_k = kc.view(torch.int16) if case["kv"] == "bf16" else kc
    view_v = vc.view(torch.int16) if case["kv"] == "bf16" else vc
    fill = nan if case["kv"] != "bf16" else np.int16(nan)
    if free.numel():
        view_k[free] = int(fill)
        view_v[free] = int(fill)
    if slots:
        s = torch.tensor(slots, dtype=torch.int64, device=kc.device)
        blk, off = s // bs, s % bs
        view_k[blk, :, off, :] = int(fill)
        view_v[blk, :, off, :] = int(fill)


def fill_fp8_cache(case):
    """Write the E4M3 case's fill rows (positions 0..ctx-1) through pkv.append."""
    dev = case["k_cache"].device
    seq = case["fill_seq"].to(dev)
    pos = case["fill_pos"].to(dev)
    bt = case["block_tables"].to(dev)
    slots = pkv.slot_mapping(bt, pos, case["k_cache"], seq_index=seq)
    ks = case["k_scale"][seq].contiguous()
    vs = case["v_scale"][seq].contiguous()
    pkv.append(case["fill_k"], case["fill_v"], slots, case["k_cache"], case["v_cache"], ks, vs)
    return slots


def run_step(case, s, split_tokens=0, out=None):
    """Append step s's new token of every sequence, then decode; returns out."""
    dev = case["k_cache"].device
    B = case["B"]
    bt = case["block_tables"].to(dev)
    ctx = case["ctx"].to(dev)
    pos = ctx.to(torch.int64) + s
    slots = pkv.slot_mapping(bt, pos, case["k_cache"])
    fp8 = case["kv"] == "e4m3"
    pkv.append(case["k_new"][s].contiguous(), case["v_new"][s].contiguous(), slots,
               case["k_cache"], case["v_cache"],
               case["k_scale"] if fp8 else None, case["v_scale"] if fp8 else None)
    lens = (ctx + s + 1).to(torch.int32)
    max_len = int(case["ctx"].max()) + s + 1 if B else 0
    return pkv.decode_attention(case["q"][s].contiguous(), case["k_cache"], case["v_cache"], bt, lens,
                                case["scale"], case["k_scale"] if fp8 else None,
                                case["v_scale"] if fp8 else None, max_context_len=max_len,
                                split_tokens=split_tokens, out=out)


def snapshot_sequence(case, b, h):
    """Raw cache words of sequence b's blocks for KV head h ([n, 1, bs, D]),
    as the generator drew them (bf16 caches; take before any append)."""
    n = case["blocks_needed"][b]
    ids = case["block_tables"][b, :n].to(torch.int64).to(case["k_cache"].device)
    k = bits16(case["k_cache"][ids][:, h:h + 1])
    v = bits16(case["v_cache"][ids][:, h:h + 1])
    return k, v


def oracle_unit(case, b, h, step, snap=None):
    """Oracle output [G, D] of query heads h*G..h*G+G-1 of sequence b after the
    appends of steps 0..step, on a one-sequence, one-head copy of the cache
    (its blocks renumbered 0..n-1, which leaves the result unchanged)."""
    bs, D = case["bs"], case["D"]
    G = case["H_q"] // case["H_kv"]
    n = case["blocks_needed"][b]
    ctx = int(case["ctx"][b])
    table = np.arange(n, dtype=np.int32)[None, :]
    if case["kv"] == "bf16":
        kc, vc = (a.copy() for a in snap)
        src, dt, ks, vs = PA.BF16, PA.BF16, None, None
        k_new = bits16(case["k_new"][:, b, h:h + 1])            # [steps, 1, D]
        v_new = bits16(case["v_new"][:, b, h:h + 1])
    else:
        kc = np.full((n, 1, bs, D), E4M3_NAN, dtype=np.uint8)
        vc = kc.copy()
        src, dt = PA.F32, PA.E4M3
        ks = case["k_scale"][b, h:h + 1].cpu().numpy()
        vs = case["v_scale"][b, h:h + 1].cpu().numpy()
        sel = (case["fill_seq"] == b).nonzero().flatten()
        rows_k = case["fill_k"][sel.to(case["fill_k"].device), h:h + 1].cpu().numpy()
        rows_v = case["fill_v"][sel.to(case["fill_v"].device), h:h + 1].cpu().numpy()
        pos = case["fill_pos"][sel].numpy()
        slots = np.array([PA.slot_of(table[0], int(p), bs) for p in pos])
        kc, vc = PA.append(rows_k, rows_v, src, slots, kc, vc, dt, ks, vs, scale_row_stride=0)
        k_new = case["k_new"][:, b, h:h + 1].cpu().numpy()
        v_new = case["v_new"][:, b, h:h + 1].cpu().numpy()
    for s in range(step + 1):
        slot = PA.slot_of(table[0], ctx + s, bs)
        kc, vc = PA.append(k_new[s][None], v_new[s][None], src, np.array([slot]), kc, vc, dt,
                           ks, vs, scale_row_stride=0)
    q = bits16(case["q"][step, b, h * G:(h + 1) * G])[None]          # [1, G, D]
    ksc = None if ks is None else ks[None, :]
    vsc = None if vs is None else vs[None, :]
    out = PA.decode_attention(q, kc, vc, dt, table, np.array([ctx + step + 1]), case["scale"],
                              ksc, vsc)
    return out[0]


def tolerance(case):
    return 2e-3 if case["kv"] == "bf16" else 5e-3
