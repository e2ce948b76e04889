"""GPU parity of multi-token (causal) query attention against the oracle:
small ragged cases over every warp arrangement and split size, the edge cases
(contexts shorter than q_len, empty contexts, q_len = 1), and sampled units
of the full-size GQA workload with four new tokens per sequence appended
through the library first."""

import numpy as np
import pytest
import torch

import paged_kv_cache_222_gb300 as pkv
import workloads as W
from oracle import paged_attention as PA

from .gpu_support import BF16_NAN, bits16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _small_case(ctxs, q_len, H_q, H_kv, D, bs, seed):
    """Paged bf16 caches holding each sequence's ctx tokens (new ones included),
    tables over a shuffled pool, NaN in every slot no sequence holds."""
    gen = torch.Generator().manual_seed(seed)
    B = len(ctxs)
    nblk = [-(-c // bs) for c in ctxs]
    mb = max(max(nblk), 1)
    pool = sum(nblk) + 5
    perm = torch.randperm(pool, generator=gen).tolist()
    table = np.full((B, mb), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        table[b, :nblk[b]] = perm[k:k + nblk[b]]
        k += nblk[b]
    kc = torch.randn((pool, H_kv, bs, D), generator=gen).to(torch.bfloat16)
    vc = torch.randn((pool, H_kv, bs, D), generator=gen).to(torch.bfloat16)
    kb, vb = kc.view(torch.int16), vc.view(torch.int16)
    used = np.zeros(pool, dtype=bool)
    for b in range(B):
        used[table[b, :nblk[b]]] = True
        for pos in range(ctxs[b], nblk[b] * bs):
            blk = int(table[b, pos // bs])
            kb[blk, :, pos % bs] = BF16_NAN
            vb[blk, :, pos % bs] = BF16_NAN
    for blk in np.nonzero(~used)[0]:
        kb[int(blk)] = BF16_NAN
        vb[int(blk)] = BF16_NAN
    q = torch.randn((B, q_len, H_q, D), generator=gen).to(torch.bfloat16)
    return dict(kc=kc, vc=vc, table=table, ctx=np.array(ctxs, dtype=np.int32), q=q, scale=D ** -0.5)


def _run(case, split_tokens=0):
    lens = torch.from_numpy(case["ctx"]).to(DEV)
    out = pkv.multi_query_attention(case["q"].to(DEV), case["kc"].to(DEV), case["vc"].to(DEV),
                                    torch.from_numpy(case["table"]).to(DEV), lens, case["scale"],
                                    max_context_len=max(int(case["ctx"].max()), 1),
                                    split_tokens=split_tokens)
    assert pkv.device_error(DEV) == 0
    return out.cpu().numpy()


def _oracle(case):
    return PA.multi_query_attention(bits16(case["q"]), bits16(case["kc"]), bits16(case["vc"]), PA.BF16,
                                    case["table"], case["ctx"], case["scale"])


@pytest.mark.parametrize("q_len,H_q,H_kv,D,bs", [
    (1, 8, 1, 128, 16),     # 8 rows: four token lanes
    (2, 8, 1, 128, 16),     # 16 rows
    (3, 10, 2, 64, 16),     # 15 rows, G = 5
    (4, 8, 1, 128, 32),     # 32 rows: the tcgen05 kernel
    (8, 4, 1, 64, 32),      # 32 rows, D = 64
    (6, 8, 1, 128, 16),     # 48 rows: a partly filled group
    (16, 8, 2, 128, 16),    # 64 rows
    (6, 3, 1, 128, 16),     # 18 rows, G = 3: the smallest tcgen05 case
    (16, 8, 1, 128, 32),    # 128 rows: the tcgen05 kernel, whole 32-token blocks per TMA box
    (12, 8, 1, 128, 16),    # 96 rows: a partly filled 128-row group
    (12, 16, 1, 128, 16),   # 192 rows: a partly filled second 128-row group
    (10, 32, 2, 64, 32),    # 160 rows, D = 64
    (16, 16, 1, 64, 16),    # 256 rows: two row blocks per head
    (14, 8, 1, 128, 16),    # 112 rows: every warp has rows, the last one only half (no idle-warp path)
    (15, 16, 1, 64, 32),    # 240 rows: a second row block of 112 rows
])
@pytest.mark.parametrize("split_tokens", [0, 64, 192])
def test_multi_query_matches_oracle(q_len, H_q, H_kv, D, bs, split_tokens):
    ctxs = [q_len, 17 + q_len, 64, 65, 300, 1000 + q_len]
    case = _small_case(ctxs, q_len, H_q, H_kv, D, bs, seed=20260200 + q_len * 7 + D + split_tokens)
    out = _run(case, split_tokens)
    want = _oracle(case)
    assert np.isfinite(out).all()
    assert np.abs(out - want).max() <= 2e-3


@pytest.mark.parametrize("scale", [-0.25, 0.0, 3.0])
@pytest.mark.parametrize("q_len,H_q", [(2, 8), (4, 8), (16, 16)])   # mma.sync; tcgen05 (32 and 256 rows)
def test_negative_zero_and_large_scales(q_len, H_q, scale):
    # the tensor-core kernel applies the logit multiplier inside the
    # exponent and folds a negative scale into Q; a zero scale gives the mean
    # of V over each query's causal range
    case = _small_case([q_len, 100, 700], q_len, H_q, 1, 128, 16, seed=20260310 + q_len)
    case["scale"] = scale
    for st in (0, 64):
        out = _run(case, st)
        want = _oracle(case)
        assert np.isfinite(out).all()
        assert np.abs(out - want).max() <= 2e-3


def test_short_and_empty_contexts_give_zeros_for_unplaced_queries():
    q_len = 8
    case = _small_case([0, 3, 8, 9], q_len, 8, 2, 128, 16, seed=20260301)
    for st in (0, 64):
        out = _run(case, st)
        want = _oracle(case)
        assert np.isfinite(out).all()
        assert np.all(out[0] == 0.0) and np.all(out[1, :5] == 0.0)
        assert np.abs(out - want).max() <= 2e-3


def test_single_query_equals_decode():
    case = _small_case([1, 40, 700, 2049], 1, 16, 2, 128, 16, seed=20260302)
    out = _run(case)
    lens = torch.from_numpy(case["ctx"]).to(DEV)
    dec = pkv.decode_attention(case["q"][:, 0].contiguous().to(DEV), case["kc"].to(DEV), case["vc"].to(DEV),
                               torch.from_numpy(case["table"]).to(DEV), lens, case["scale"],
                               max_context_len=2049)
    assert np.abs(out[:, 0] - dec.cpu().numpy()).max() <= 1e-4


def test_split_count_does_not_change_the_result():
    case = _small_case([5000, 333, 4096], 4, 32, 4, 128, 16, seed=20260303)
    outs = [_run(case, st) for st in (64, 256, 1024, 4096, 16384)]
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-5


@pytest.mark.parametrize("q_len", [2, 3, 4, 8, 16])   # mma.sync; persistent tcgen05 (24 .. 128 rows)
def test_full_size_gqa_workload_every_unit(q_len):
    """B=64, H_q=64, H_kv=8, D=128, bs=16, contexts U[512, 8192]: the q_len
    new tokens of every sequence are appended by pkv.append, then attended
    causally; all 512 (sequence, KV head) units are checked against the
    oracle (run on the host cores from the generator's inputs)."""
    from tests import oracle_pool as OP
    case = W.make_case("gqa_bf16", device=DEV, steps=q_len)
    src = OP.UnitSource(case)
    bt = case["block_tables"].to(DEV)
    ctx = case["ctx"].to(DEV).to(torch.int64)
    for s in range(q_len):
        slots = pkv.slot_mapping(bt, ctx + s, case["k_cache"])
        pkv.append(case["k_new"][s].contiguous(), case["v_new"][s].contiguous(), slots,
                   case["k_cache"], case["v_cache"])
    lens = (ctx + q_len).to(torch.int32)
    q = case["q"].permute(1, 0, 2, 3).contiguous()                          # [B, q_len, H_q, D]
    out = pkv.multi_query_attention(q, case["k_cache"], case["v_cache"], bt, lens, case["scale"],
                                    max_context_len=int(lens.max()))
    assert pkv.device_error(DEV) == 0
    out = out.cpu().numpy()
    assert np.isfinite(out).all()
    units = [(b, h) for b in range(case["B"]) for h in range(case["H_kv"])]
    res = OP.run_units(src, units, q_len, list(range(q_len)))
    assert res["units"] == 512
    assert OP.max_abs_err(out, res["outputs"], case["H_q"] // case["H_kv"], multi=True) <= 2e-3


@pytest.mark.parametrize("q_len,H_q,H_kv", [(8, 16, 1), (16, 8, 1)])
def test_tcgen05_path_short_and_empty_contexts(q_len, H_q, H_kv):
    case = _small_case([0, 3, q_len, q_len + 1, 70, 1100], q_len, H_q, H_kv, 128, 16, seed=20260304 + q_len)
    for st in (0, 64, 320):
        out = _run(case, st)
        want = _oracle(case)
        assert np.isfinite(out).all()
        assert np.all(out[0] == 0.0) and np.all(out[1, :q_len - 3] == 0.0)
        assert np.abs(out - want).max() <= 2e-3


def test_tcgen05_split_count_does_not_change_the_result():
    case = _small_case([5000, 333, 4096], 16, 64, 8, 128, 16, seed=20260305)
    outs = [_run(case, st) for st in (64, 256, 1024, 4096, 16384)]
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-5


def test_tcgen05_many_units_per_cta_full_size():
    """The GQA workload (B=64, H_kv=8, contexts up to 8208) with 256-token
    splits: about 16,900 work units, some 110 per persistent CTA, so the ring
    of published units wraps many times and partials of 33 splits are
    combined.  Same result as the default plan (one split per sequence)."""
    q_len = 16
    case = W.make_case("gqa_bf16", device=DEV, steps=q_len)
    bt = case["block_tables"].to(DEV)
    lens = (case["ctx"] + q_len).to(DEV).to(torch.int32)
    q = case["q"].permute(1, 0, 2, 3).contiguous()
    mx = int(lens.max())
    plan = pkv.multi_query_plan(case["B"], q_len, case["H_q"], case["k_cache"], mx, 256, 152)
    assert plan.workers == 0 and plan.max_splits == -(-mx // 256)
    a = pkv.multi_query_attention(q, case["k_cache"], case["v_cache"], bt, lens, case["scale"], mx)
    b = pkv.multi_query_attention(q, case["k_cache"], case["v_cache"], bt, lens, case["scale"], mx,
                                  split_tokens=256)
    assert pkv.device_error(DEV) == 0
    assert np.abs(a.cpu().numpy() - b.cpu().numpy()).max() <= 1e-5


def test_tcgen05_under_graph_capture_and_on_two_streams():
    """The persistent kernel's unit counter and order live in each call's
    workspace: two calls at once on two streams, and a captured call
    replayed from a CUDA graph, give the eager result bit for bit."""
    case = _small_case([700, 33, 4100, 1, 1500], 16, 16, 2, 128, 16, seed=20260712)
    dev = torch.device(DEV)
    q, kc, vc = case["q"].to(dev), case["kc"].to(dev), case["vc"].to(dev)
    tbl = torch.from_numpy(case["table"]).to(dev)
    lens = torch.from_numpy(case["ctx"]).to(dev)
    mx = int(case["ctx"].max())
    plan = pkv.multi_query_plan(q.shape[0], q.shape[1], q.shape[2], kc, mx, 256, 152)
    assert plan.workers == 0

    def call(out, ws):
        return pkv.multi_query_attention(q, kc, vc, tbl, lens, case["scale"], mx, split_tokens=256, out=out,
                                         workspace=ws)

    want = call(None, None).cpu()
    outs = [torch.empty(q.shape, dtype=torch.float32, device=dev) for _ in range(3)]
    wss = [torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=dev) for _ in range(3)]
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        call(outs[0], wss[0])
    with torch.cuda.stream(s2):
        call(outs[1], wss[1])
    torch.cuda.current_stream().wait_stream(s1)
    torch.cuda.current_stream().wait_stream(s2)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].cpu(), want) and torch.equal(outs[1].cpu(), want)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(outs[2], wss[2])
    outs[2].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs[2].cpu(), want)
    assert pkv.device_error(DEV) == 0
    assert np.abs(want.numpy() - _oracle(case)).max() <= 2e-3
