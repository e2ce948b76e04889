"""GPU parity at the largest batch the calls take (65,535 sequences: the decode
and mma.sync multi-token grids put the sequence on the grid's z axis, whose
limit that is).  Sampled units are compared with the float64 oracle; the whole
output is checked through properties that hold at any size (every row finite,
the split count changes nothing)."""

import numpy as np
import pytest
import torch

import paged_kv_cache_222_gb300 as pkv
import workloads as W
from oracle import paged_attention as PA
from tests import gpu_support as S

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
B_MAX = 65535
SAMPLED = (0, 1, 2, 4095, 32767, 65533, 65534)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_222_gb300 import build
    build.build()
    pkv.library()
    assert pkv.device_error(DEV) == 0
    yield
    assert pkv.device_error(DEV) == 0


def test_host_rejects_one_sequence_more():
    kc = torch.zeros((4, 1, 16, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(Exception):
        pkv.decode_plan(B_MAX + 1, 4, kc, 16)


def test_decode_at_the_largest_batch():
    spec = dict(B=B_MAX, H_q=4, H_kv=1, D=64, bs=16, kv="bf16", free_frac=0.25, steps=1, seed=65,
                q_mult=1.0, ctx_range=(0, 200))
    case = W.make_case(spec, device=DEV)
    S.poison_unused(case)
    snaps = {(b, 0): S.snapshot_sequence(case, b, 0) for b in SAMPLED}
    out0 = S.run_step(case, 0, split_tokens=0)
    out64 = S.run_step(case, 0, split_tokens=64)   # up to four 64-token splits per sequence
    plan = pkv.decode_plan(B_MAX, 4, case["k_cache"], int(case["ctx"].max()) + 1, split_tokens=64)
    assert plan.max_splits >= 3
    dev = case["k_cache"].device
    lens = (case["ctx"] + 1).to(torch.int32).to(dev)
    fused = pkv.decode_attention(case["q"][0].contiguous(), case["k_cache"], case["v_cache"],
                                 case["block_tables"].to(dev), lens, case["scale"], max_context_len=int(lens.max()),
                                 k_new=case["k_new"][0].contiguous(), v_new=case["v_new"][0].contiguous())
    assert pkv.device_error(DEV) == 0
    assert torch.equal(out0, fused)                 # the one-launch step, same plan
    assert bool(torch.isfinite(out0).all()) and bool(torch.isfinite(out64).all())
    assert float((out0 - out64).abs().max()) < 1e-5
    got = out0.cpu().numpy()
    for b in SAMPLED:
        ref = S.oracle_unit(case, b, 0, 0, snaps[(b, 0)])
        assert np.max(np.abs(got[b] - ref)) <= 2e-3, b


def _big_mq_case(q_len, H_q, H_kv, D, bs, ctx_hi, seed):
    """B_MAX sequences of q_len..ctx_hi tokens (new ones included) in a shuffled
    pool, NaN in every slot past a sequence's end and in every free block."""
    gen = torch.Generator().manual_seed(seed)
    ctx = torch.randint(q_len, ctx_hi + 1, (B_MAX,), generator=gen)
    nblk = (ctx + bs - 1) // bs
    mb = int(nblk.max())
    pool = int(nblk.sum()) + 5
    perm = torch.randperm(pool, generator=gen)
    off = torch.cumsum(nblk, 0) - nblk
    j = torch.arange(mb)
    held = j[None, :] < nblk[:, None]
    table = torch.where(held, perm[(off[:, None] + j[None, :]).clamp(max=pool - 1)], torch.full((1,), -1))
    kc = torch.randn((pool, H_kv, bs, D), generator=gen).to(torch.bfloat16)
    vc = torch.randn((pool, H_kv, bs, D), generator=gen).to(torch.bfloat16)
    kb, vb = kc.view(torch.int16), vc.view(torch.int16)
    pos = torch.arange(mb * bs)
    tail = (pos[None, :] >= ctx[:, None]) & (pos[None, :] < (nblk * bs)[:, None])
    rows, cols = tail.nonzero(as_tuple=True)
    blk = table[rows, cols // bs]
    kb[blk, :, cols % bs] = S.BF16_NAN
    vb[blk, :, cols % bs] = S.BF16_NAN
    free = torch.ones(pool, dtype=torch.bool)
    free[table[held]] = False
    kb[free] = S.BF16_NAN
    vb[free] = S.BF16_NAN
    q = torch.randn((B_MAX, q_len, H_q, D), generator=gen).to(torch.bfloat16)
    return dict(kc=kc, vc=vc, table=table.to(torch.int32).numpy(), ctx=ctx.to(torch.int32).numpy(), q=q,
                scale=D ** -0.5)


@pytest.mark.parametrize("q_len,H_q,H_kv,D,bs", [
    (2, 4, 1, 64, 16),      # 8 rows: the mma.sync kernel (sequence on the grid's z axis)
    (4, 8, 1, 64, 32),      # 32 rows: the persistent tcgen05 kernel, 65,535 units per split
])
def test_multi_query_at_the_largest_batch(q_len, H_q, H_kv, D, bs):
    case = _big_mq_case(q_len, H_q, H_kv, D, bs, ctx_hi=100, seed=66 + q_len)
    lens = torch.from_numpy(case["ctx"]).to(DEV)
    table = torch.from_numpy(case["table"]).to(DEV)
    q, kc, vc = case["q"].to(DEV), case["kc"].to(DEV), case["vc"].to(DEV)
    mx = int(case["ctx"].max())
    outs = [pkv.multi_query_attention(q, kc, vc, table, lens, case["scale"], max_context_len=mx,
                                      split_tokens=st) for st in (0, 64)]
    assert pkv.device_error(DEV) == 0
    for o in outs:
        assert bool(torch.isfinite(o).all())
    # Splits change each row's running maximum, so every probability is
    # rounded into its bf16 hi + lo pair (about 2^-17 relative) from a
    # different value: the two results may differ by up to ~2 * 2^-17 *
    # max |v - out|, about 1e-4 for N(0, 1) values over at most 100 tokens.
    # (Three sequences stay within 1e-5; 65,535 reach 1.3e-5.)
    assert float((outs[0] - outs[1]).abs().max()) < 1e-4
    sel = np.array(SAMPLED)
    ref = PA.multi_query_attention(S.bits16(case["q"][torch.from_numpy(sel)]), S.bits16(case["kc"]),
                                   S.bits16(case["vc"]), PA.BF16, case["table"][sel], case["ctx"][sel],
                                   case["scale"])
    got = outs[0].cpu().numpy()[sel]
    assert np.max(np.abs(got - ref)) <= 2e-3


def test_decode_over_a_million_tokens():
    """One sequence of 2^20 + 1 tokens after the append, beside a short one,
    8 KV heads: the pool's block ids pass 65,536 and cache byte offsets pass
    2^31 (32 KB per block).  Append + decode and the fused one-launch step
    agree bit for bit; units of the last head (the largest offsets), the
    first head and the short sequence match the oracle."""
    spec = dict(B=2, H_q=64, H_kv=8, D=128, bs=16, kv="bf16", free_frac=0.25, steps=1, seed=67,
                q_mult=1.0, ctx=(1 << 20, 300))
    case = W.make_case(spec, device=DEV)
    kc = case["k_cache"]
    assert kc.shape[0] * kc[0].numel() * kc.element_size() > 1 << 31
    S.poison_unused(case)
    units = [(0, 0), (0, 7), (1, 3)]
    snaps = {u: S.snapshot_sequence(case, *u) for u in units}
    out = S.run_step(case, 0)
    dev = kc.device
    lens = (case["ctx"] + 1).to(torch.int32).to(dev)
    assert int(lens[0]) == (1 << 20) + 1 and int(case["block_tables"].max()) >= 65536
    fused = pkv.decode_attention(case["q"][0].contiguous(), kc, case["v_cache"], case["block_tables"].to(dev),
                                 lens, case["scale"], max_context_len=int(lens.max()),
                                 k_new=case["k_new"][0].contiguous(), v_new=case["v_new"][0].contiguous())
    assert pkv.device_error(DEV) == 0
    assert torch.equal(out, fused)
    got = out.cpu().numpy()
    G = 8
    for b, h in units:
        ref = S.oracle_unit(case, b, h, 0, snaps[(b, h)])
        assert np.max(np.abs(got[b, h * G:(h + 1) * G] - ref)) <= 2e-3, (b, h)


def test_fp8_decode_at_the_largest_batch():
    """E4M3 caches at 65,535 sequences: the fill (every position through
    pkv_append with per-(sequence, head) scales, row b * stride + h up to
    sequence 65,534), then decode with one split and with 64-token splits.
    P enters P.V as one f16 term, so splits move results by up to the FP8
    tolerance; both are checked against the oracle on sampled units, every
    row for finiteness, and the fused step against the two-call step."""
    spec = dict(B=B_MAX, H_q=4, H_kv=1, D=64, bs=16, kv="e4m3", free_frac=0.25, steps=1, seed=68,
                q_mult=1.0, ctx_range=(0, 200))
    case = W.make_case(spec, device=DEV)
    case["k_cache"].fill_(S.E4M3_NAN)
    case["v_cache"].fill_(S.E4M3_NAN)
    S.fill_fp8_cache(case)
    outs = [S.run_step(case, 0, split_tokens=st) for st in (0, 64)]
    dev = case["k_cache"].device
    lens = (case["ctx"] + 1).to(torch.int32).to(dev)
    fused = pkv.decode_attention(case["q"][0].contiguous(), case["k_cache"], case["v_cache"],
                                 case["block_tables"].to(dev), lens, case["scale"], case["k_scale"],
                                 case["v_scale"], max_context_len=int(lens.max()),
                                 k_new=case["k_new"][0].contiguous(), v_new=case["v_new"][0].contiguous())
    assert pkv.device_error(DEV) == 0
    assert torch.equal(outs[0], fused)
    for o in outs:
        assert bool(torch.isfinite(o).all())
        got = o.cpu().numpy()
        for b in SAMPLED:
            ref = S.oracle_unit(case, b, 0, 0)
            assert np.max(np.abs(got[b] - ref)) <= S.tolerance(case), b
