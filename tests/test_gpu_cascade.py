"""Cascade (shared-prefix) decode on the GPU: parity with the oracle and with
the plain decode path on batches whose sequences share their first tokens."""

import numpy as np
import pytest
import torch

import paged_kv_cache_222_gb300 as pkv
import workloads as W
from tests import gpu_support as S

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_222_gb300 import build
    build.build()
    pkv.library()
    assert pkv.device_error(DEV) == 0
    yield
    assert pkv.device_error(DEV) == 0


def shared_case(B, prefix, suffix_range, G, H_kv, D, bs, seed, q_mult=1.0):
    spec = dict(B=B, prefix=prefix, suffix_range=suffix_range, H_q=G * H_kv, H_kv=H_kv, D=D, bs=bs,
                kv="bf16", free_frac=0.1, steps=1, seed=seed, q_mult=q_mult)
    return W.make_case(spec, device=DEV)


def run_cascade(case):
    dev = DEV
    B, bs = case["B"], case["bs"]
    bt = case["block_tables"].to(dev)
    ctx = case["ctx"].to(dev)
    slots = pkv.slot_mapping(bt, ctx.to(torch.int64), case["k_cache"])
    pkv.append(case["k_new"][0].contiguous(), case["v_new"][0].contiguous(), slots, case["k_cache"],
               case["v_cache"])
    lens = (ctx + 1).to(torch.int32)
    mx = int(case["ctx"].max()) + 1
    prefix = case["prefix"]
    pblocks = bt[0, : prefix // bs].contiguous()
    out_c = pkv.cascade_decode_attention(case["q"][0].contiguous(), case["k_cache"], case["v_cache"],
                                         pblocks, prefix, bt, lens, case["scale"], mx)
    out_p = pkv.decode_attention(case["q"][0].contiguous(), case["k_cache"], case["v_cache"], bt, lens,
                                 case["scale"], max_context_len=mx)
    return out_c, out_p


@pytest.mark.parametrize("B,prefix,suffix,G,H_kv,D,bs", [
    (5, 64, (1, 300), 8, 2, 128, 16),
    (3, 128, (1, 100), 8, 1, 128, 32),
    (7, 48, (1, 50), 4, 2, 64, 16),        # prefix not a multiple of the 64-token tile
    (2, 512, (1, 40), 16, 2, 128, 32),     # G = 16
    (33, 96, (1, 20), 6, 1, 64, 32),       # ragged row blocks (33 * 6 rows)
    (64, 256, (1, 2000), 8, 2, 128, 16),   # long suffixes: the plan takes one prefix range
    (16, 128, (1, 3000), 8, 1, 128, 16),   # two one-tile ranges beside long suffixes
    (4, 256, (1, 1000), 8, 2, 128, 16),    # 8 slots per row: 4 suffix splits + 4 prefix ranges
    (8, 192, (1, 900), 8, 2, 64, 16),      # 5-8 slots per row, D = 64
    (50, 128, (1, 100), 6, 1, 64, 32),     # sequence 42's rows straddle two prefix row blocks
    (100, 64, (1, 700), 3, 2, 128, 16),    # G = 3: several straddling sequences, several splits
])
def test_cascade_matches_oracle_and_plain_decode(B, prefix, suffix, G, H_kv, D, bs):
    case = shared_case(B, prefix, suffix, G, H_kv, D, bs, seed=500 + B + prefix)
    S.poison_unused(case)
    snaps = {(b, h): S.snapshot_sequence(case, b, h) for b in range(B) for h in range(H_kv)}
    out_c, out_p = run_cascade(case)
    got = out_c.cpu().numpy()
    for (b, h), snap in snaps.items():
        ref = S.oracle_unit(case, b, h, 0, snap)
        assert np.max(np.abs(got[b, h * G:(h + 1) * G] - ref)) <= 2e-3
    assert torch.max(torch.abs(out_c - out_p)) < 1e-4


@pytest.mark.parametrize("B,prefix,suffix,G,H_kv,D,bs,ranges,range_tokens", [
    (128, 16384, (1, 300), 8, 8, 128, 16, 4, 4096),   # ranges at their 256-block cap; 5 slots per row
    (4, 16384, (1, 500), 8, 2, 128, 16, 64, 256),     # 64 ranges: 66 slots per row, the generic combine
    (3, 40960, (1, 64), 4, 1, 64, 32, 64, 640),       # D = 64, 32-token blocks, 65 slots per row
])
def test_cascade_long_prefixes(B, prefix, suffix, G, H_kv, D, bs, ranges, range_tokens):
    case = shared_case(B, prefix, suffix, G, H_kv, D, bs, seed=1500 + B)
    S.poison_unused(case)
    mx = int(case["ctx"].max()) + 1
    plan = pkv.cascade_plan(B, G * H_kv, case["k_cache"], prefix, mx)
    assert plan.workers == ranges and plan.prefix_split_tokens == range_tokens
    units = [(b, h) for b in sorted({0, B // 2, B - 1}) for h in sorted({0, H_kv - 1})]
    snaps = {u: S.snapshot_sequence(case, *u) for u in units}
    out_c, out_p = run_cascade(case)
    assert pkv.device_error(DEV) == 0
    got = out_c.cpu().numpy()
    for (b, h), snap in snaps.items():
        ref = S.oracle_unit(case, b, h, 0, snap)
        assert np.max(np.abs(got[b, h * G:(h + 1) * G] - ref)) <= 2e-3
    assert torch.max(torch.abs(out_c - out_p)) < 1e-4   # every unit, against the plain decode


@pytest.mark.parametrize("scale", [-0.3, 0.0, 2.5])
def test_cascade_negative_zero_and_large_scales(scale):
    # the prefix kernel applies the logit multiplier inside the exponent and
    # folds a negative scale into Q; a zero scale gives the mean of V
    B, G, H_kv = 5, 8, 2
    case = shared_case(B, 128, (1, 300), G, H_kv, 128, 16, seed=733)
    case["scale"] = scale
    S.poison_unused(case)
    snaps = {(b, h): S.snapshot_sequence(case, b, h) for b in range(B) for h in range(H_kv)}
    out_c, out_p = run_cascade(case)
    got = out_c.cpu().numpy()
    assert np.isfinite(got).all()
    for (b, h), snap in snaps.items():
        ref = S.oracle_unit(case, b, h, 0, snap)
        assert np.max(np.abs(got[b, h * G:(h + 1) * G] - ref)) <= 2e-3
    assert torch.max(torch.abs(out_c - out_p)) < 1e-4


@pytest.mark.parametrize("B,prefix,suffix,G,H_kv,D,bs,every", [
    (12, 128, (1, 200), 8, 2, 128, 16, 3),    # one suffix split per sequence
    (9, 64, (1, 700), 4, 2, 64, 16, 3),       # several suffix splits
    (8, 192, (1, 900), 8, 2, 128, 16, 3),     # 7 slots per row
    (6, 128, (1, 200), 8, 2, 128, 16, 1),     # no sequence has a private token
])
def test_cascade_sequences_that_attend_only_the_prefix(B, prefix, suffix, G, H_kv, D, bs, every):
    """Every `every`-th sequence attends exactly the shared prefix (no private
    token): its suffix slots are never written, and the workspace is filled
    with NaN first, so a combine that read them would show it."""
    from oracle import paged_attention as PA
    case = shared_case(B, prefix, suffix, G, H_kv, D, bs, seed=900 + B + D)
    S.poison_unused(case)
    bt = case["block_tables"].to(DEV)
    lens = case["ctx"].clone().to(torch.int32)
    lens[::every] = prefix
    mx = int(lens.max())
    q = case["q"][0].contiguous()
    pblocks = bt[0, : prefix // bs].contiguous()
    plan = pkv.cascade_plan(B, G * H_kv, case["k_cache"], prefix, mx)
    ws = torch.full((int(plan.workspace_bytes),), 0xFF, dtype=torch.uint8, device=DEV)
    out_c = pkv.cascade_decode_attention(q, case["k_cache"], case["v_cache"], pblocks, prefix, bt,
                                         lens.to(DEV), case["scale"], mx, workspace=ws)
    got = out_c.cpu().numpy()
    lens_h = lens.numpy()
    for b in range(B):
        n = case["blocks_needed"][b]
        for h in range(H_kv):
            k, v = S.snapshot_sequence(case, b, h)
            want = PA.decode_attention(S.bits16(q[b, h * G:(h + 1) * G])[None], k, v, PA.BF16,
                                       np.arange(n, dtype=np.int32)[None, :], lens_h[b:b + 1],
                                       case["scale"])[0]
            assert np.max(np.abs(got[b, h * G:(h + 1) * G] - want)) <= 2e-3, (b, h, int(lens_h[b]))


def test_cascade_full_size_shared_prefix_workload_every_unit():
    """B=128 sequences sharing 4096 tokens (128 blocks of 32) plus private
    suffixes of U[64, 1024]: all 1024 (sequence, KV head) units against the
    oracle's plain decode of each whole sequence, and against the plain
    decode call."""
    from tests import oracle_pool as OP
    case = W.make_case("shared_prefix", device=DEV)
    src = OP.UnitSource(case)
    out_c, out_p = run_cascade(case)
    assert torch.max(torch.abs(out_c - out_p)) < 1e-4
    got = out_c.cpu().numpy()
    units = [(b, h) for b in range(case["B"]) for h in range(case["H_kv"])]
    res = OP.run_units(src, units, 1, [0])
    assert res["units"] == 1024
    assert OP.max_abs_err(got, res["outputs"], case["H_q"] // case["H_kv"]) <= 2e-3


def test_cascade_sequence_shorter_than_the_prefix_is_recorded():
    """A cascade call's sequences must each hold the whole shared prefix: one
    that is shorter is reported in the device error word (the prefix kernel
    attends the prefix for every row); a correct call afterwards reports
    nothing."""
    case = shared_case(4, 128, (1, 100), 8, 2, 128, 16, seed=4242)
    bt = case["block_tables"].to(DEV)
    lens = (case["ctx"] + 1).to(torch.int32)
    mx = int(lens.max())
    pblocks = bt[0, :128 // 16].contiguous()
    q = case["q"][0].contiguous()
    short = lens.clone()
    short[2] = 128 - 5
    pkv.cascade_decode_attention(q, case["k_cache"], case["v_cache"], pblocks, 128, bt, short.to(DEV),
                                 case["scale"], mx)
    assert pkv.device_error(DEV) == 3
    out = pkv.cascade_decode_attention(q, case["k_cache"], case["v_cache"], pblocks, 128, bt, lens.to(DEV),
                                       case["scale"], mx)
    assert pkv.device_error(DEV) == 0
    assert torch.all(torch.isfinite(out))


def test_cascade_sharp_softmax():
    case = shared_case(4, 1024, (100, 600), 8, 2, 128, 32, seed=77, q_mult=4.0)
    snaps = {(b, h): S.snapshot_sequence(case, b, h) for b in range(4) for h in range(2)}
    out_c, out_p = run_cascade(case)
    got = out_c.cpu().numpy()
    for (b, h), snap in snaps.items():
        ref = S.oracle_unit(case, b, h, 0, snap)
        assert np.max(np.abs(got[b, h * 8:(h + 1) * 8] - ref)) <= 2e-3


def test_cascade_under_graph_capture_and_on_two_streams():
    """The call forks its suffix decode onto the library's side stream and
    joins it back: captured into a CUDA graph and replayed, and issued on two
    streams at once, it gives the eager result bit for bit."""
    case = shared_case(9, 256, (1, 200), 8, 2, 128, 16, seed=20260711)
    out_c, _ = run_cascade(case)                      # appends the new token, eager result
    bs = case["bs"]
    bt = case["block_tables"].to(DEV)
    lens = (case["ctx"].to(DEV) + 1).to(torch.int32)
    mx = int(case["ctx"].max()) + 1
    prefix = case["prefix"]
    pblocks = bt[0, : prefix // bs].contiguous()
    q = case["q"][0].contiguous()
    plan = pkv.cascade_plan(q.shape[0], q.shape[1], pkv.cache_desc(case["k_cache"]), prefix, mx)

    def call(out, ws):
        return pkv.cascade_decode_attention(q, case["k_cache"], case["v_cache"], pblocks, prefix, bt, lens,
                                            case["scale"], mx, out=out, workspace=ws)

    want = out_c.cpu()
    outs = [torch.empty_like(out_c) for _ in range(3)]
    wss = [torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=DEV) for _ in range(3)]
    s1, s2 = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
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


def test_cascade_calls_sharing_one_workspace():
    """Back-to-back calls on one workspace (filled with garbage first), with
    lengths that alternate between two sets (some sequences with no private
    token), each give the plain decode's result: no piece of an earlier call
    leaks into a later one."""
    case = shared_case(40, 128, (1, 600), 8, 2, 128, 16, seed=31337)
    out_c, out_p = run_cascade(case)                  # appends the new token
    bs = case["bs"]
    bt = case["block_tables"].to(DEV)
    lens = (case["ctx"].to(DEV) + 1).to(torch.int32)
    mx = int(case["ctx"].max()) + 1
    prefix = case["prefix"]
    pblocks = bt[0, : prefix // bs].contiguous()
    q = case["q"][0].contiguous()
    plan = pkv.cascade_plan(q.shape[0], q.shape[1], pkv.cache_desc(case["k_cache"]), prefix, mx)
    ws = torch.full((int(plan.workspace_bytes),), 0x7F, dtype=torch.uint8, device=DEV)
    short = torch.clamp(lens - 37, min=prefix).to(torch.int32)   # fewer private tokens, some none
    for ln in (lens, short, lens, short):
        got = pkv.cascade_decode_attention(q, case["k_cache"], case["v_cache"], pblocks, prefix, bt, ln,
                                           case["scale"], mx, workspace=ws)
        want = pkv.decode_attention(q, case["k_cache"], case["v_cache"], bt, ln, case["scale"], max_context_len=mx)
        assert torch.max(torch.abs(got - want)) < 1e-4
    assert torch.max(torch.abs(out_c - out_p)) < 1e-4
    assert pkv.device_error(DEV) == 0
