"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Append and E4M3 quantisation must be bit-exact; decode must be within max-abs
2e-3 (bf16 KV) or 5e-3 (E4M3 KV, against the oracle's identically dequantised
values) over every output compared.
"""

import math

import numpy as np
import pytest
import torch

import paged_kv_cache_222_gb300 as pkv
import workloads as W
from oracle import formats as F
from oracle import paged_attention as PA
from tests import gpu_support as S
from tests import oracle_pool as OP

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


def small_case(kv="bf16", D=128, G=8, H_kv=2, bs=16, B=3, ctx_range=(1, 300), steps=1, seed=7,
               q_mult=1.0, ctx=None):
    spec = dict(B=B, H_q=G * H_kv, H_kv=H_kv, D=D, bs=bs, kv=kv, free_frac=0.25, steps=steps,
                seed=seed, q_mult=q_mult)
    if ctx is not None:
        spec["ctx"] = tuple(ctx)
    else:
        spec["ctx_range"] = ctx_range
    return W.make_case(spec, device=DEV)


def check_all_units(case, out, step=0, snaps=None):
    G = case["H_q"] // case["H_kv"]
    got = out.cpu().numpy()
    worst = 0.0
    for b in range(case["B"]):
        for h in range(case["H_kv"]):
            ref = S.oracle_unit(case, b, h, step, None if snaps is None else snaps[(b, h)])
            err = np.max(np.abs(got[b, h * G:(h + 1) * G] - ref))
            worst = max(worst, float(err))
    assert worst <= S.tolerance(case), worst
    return worst


def snaps_for(case, units=None):
    if case["kv"] != "bf16":
        return None
    units = units or [(b, h) for b in range(case["B"]) for h in range(case["H_kv"])]
    return {(b, h): S.snapshot_sequence(case, b, h) for b, h in units}


# ------------------------------------------------------------------ append


def test_append_bf16_copies_bits_exactly():
    case = small_case(kv="bf16", D=64, H_kv=2, bs=16, B=5, ctx_range=(3, 60))
    k0, v0 = S.bits16(case["k_cache"]), S.bits16(case["v_cache"])
    n = 40
    g = torch.Generator(device=DEV).manual_seed(3)
    kn = torch.randn((n, 2, 64), generator=g, device=DEV).to(torch.bfloat16)
    vn = torch.randn((n, 2, 64), generator=g, device=DEV).to(torch.bfloat16)
    slots = torch.randperm(case["num_blocks"] * 16, device=DEV)[:n]
    slots[3] = -1
    slots[17] = -5
    pkv.append(kn, vn, slots, case["k_cache"], case["v_cache"])
    k1, v1 = PA.append(S.bits16(kn), S.bits16(vn), PA.BF16, slots.cpu().numpy(), k0, v0, PA.BF16)
    assert np.array_equal(S.bits16(case["k_cache"]), k1)
    assert np.array_equal(S.bits16(case["v_cache"]), v1)


@pytest.mark.parametrize("src,dst,per_row", [("f32", "e4m3", True), ("bf16", "e4m3", True),
                                             ("f32", "e4m3", False), ("f32", "bf16", True)])
def test_append_quantise_bit_exact(src, dst, per_row):
    nb, H, bs, D, n = 24, 4, 32, 128, 300
    g = torch.Generator(device=DEV).manual_seed(11)
    x = torch.randn((n, H, D), generator=g, device=DEV) * 3
    y = torch.randn((n, H, D), generator=g, device=DEV) * 3
    x[0, 0, :4] = torch.tensor([1e9, -1e9, 0.0, -0.0])
    if src == "bf16":
        x, y = x.to(torch.bfloat16), y.to(torch.bfloat16)
    cdt = torch.uint8 if dst == "e4m3" else torch.bfloat16
    kc = torch.zeros((nb, H, bs, D), dtype=cdt, device=DEV)
    vc = torch.zeros_like(kc)
    slots = torch.randperm(nb * bs, device=DEV)[:n]
    ks = vs = None
    if dst == "e4m3":
        shape = (n, H) if per_row else (H,)
        ks = (torch.rand(shape, generator=g, device=DEV) * 0.02 + 0.003).contiguous()
        vs = (torch.rand(shape, generator=g, device=DEV) * 0.02 + 0.003).contiguous()
    pkv.append(x, y, slots, kc, vc, ks, vs)
    xs = S.bits16(x) if src == "bf16" else x.cpu().numpy()
    ys = S.bits16(y) if src == "bf16" else y.cpu().numpy()
    raw = (lambda t: S.bits16(t)) if dst == "bf16" else (lambda t: S.bytes8(t))
    k0 = raw(torch.zeros_like(kc))
    stride = (H if per_row else 0) if dst == "e4m3" else 0
    k1, v1 = PA.append(xs, ys, PA.BF16 if src == "bf16" else PA.F32, slots.cpu().numpy(), k0, k0.copy(),
                       PA.E4M3 if dst == "e4m3" else PA.BF16,
                       None if ks is None else ks.cpu().numpy(), None if vs is None else vs.cpu().numpy(),
                       scale_row_stride=stride)
    assert np.array_equal(raw(kc), k1)
    assert np.array_equal(raw(vc), v1)


def _sweep_values():
    """fp32 values covering every exponent and the E4M3 rounding boundaries."""
    sign = np.array([0, 1], dtype=np.uint32) << 31
    exps = np.arange(256, dtype=np.uint32) << 23
    top = np.arange(8, dtype=np.uint32) << 20                    # the 3 kept mantissa bits
    low = np.array([0, 1, 0x7FFFF, 0x80000, 0x80001, 0xFFFFF, 0x3FFFF, 0xC0000], dtype=np.uint32)
    grid = (sign[:, None, None, None] | exps[None, :, None, None] | top[None, None, :, None]
            | low[None, None, None, :]).ravel()
    pos = F.E4M3_VALUES[:0x7F]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0)),
                           pos.astype(np.float32)])
    rng = np.random.default_rng(5)
    rand = np.concatenate([(rng.standard_normal(1 << 18) * 100).astype(np.float32),
                           rng.integers(0, 1 << 32, 1 << 18, dtype=np.uint64).astype(np.uint32).view(np.float32)])
    vals = np.concatenate([grid.view(np.float32), near, -near, rand])
    pad = (-vals.size) % 128
    return np.concatenate([vals, np.zeros(pad, dtype=np.float32)])


@pytest.mark.parametrize("scale", [1.0, 0.0087890625, 0.0123])
def test_e4m3_quantisation_sweep(scale):
    vals = _sweep_values()
    n = vals.size // 128
    x = torch.from_numpy(vals.reshape(n, 1, 128)).to(DEV)
    kc = torch.zeros((n, 1, 16, 128), dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    slots = torch.arange(n, device=DEV, dtype=torch.int64) * 16
    sc = torch.full((1,), scale, dtype=torch.float32, device=DEV)
    pkv.append(x, x, slots, kc, vc, sc, sc)
    got = S.bytes8(kc[:, 0, 0, :]).reshape(-1)
    want = F.e4m3_encode(F.f32_div(vals, np.float32(scale)))
    nan = np.isnan(vals)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7F) == 0x7F)        # NaN stays NaN


def _oracle_code_steps(scale):
    """Where the oracle's quantiser (fp32 division by `scale`, then the
    brute-force E4M3 encoder) changes code over the non-negative finite fp32
    bit patterns 0 .. 0x7F800000 (+inf), in pattern order: (first pattern of
    each new code, that code).  The composition is monotone in the pattern,
    so one bisection per code finds its first pattern."""
    enc = lambda u: F.e4m3_encode(F.f32_div(np.asarray(u, dtype=np.uint32).view(np.float32), np.float32(scale)))
    codes = np.arange(1, 0x7F, dtype=np.int64)
    lo = np.zeros(codes.size, dtype=np.int64)                  # enc(lo) < code
    hi = np.full(codes.size, 0x7F800000, dtype=np.int64)       # enc(hi) >= code
    assert np.all(enc(lo) < codes) and np.all(enc(hi) >= codes)
    while np.any(hi - lo > 1):
        mid = (lo + hi) // 2
        up = enc(mid).astype(np.int64) >= codes
        hi = np.where(up, mid, hi)
        lo = np.where(up, lo, mid)
    first = np.unique(hi)
    return first, enc(first).astype(np.int64)


@pytest.mark.parametrize("scale", [1.0, 0.0123])
def test_e4m3_quantisation_every_fp32_pattern(scale):
    """All 2^32 fp32 bit patterns through the append kernel: the positive
    half must step through the codes exactly where the oracle does, NaN
    patterns stay NaN, and each negative pattern gives its magnitude's code
    with the sign bit set."""
    n_fin = 0x7F800001                          # +0 .. +inf
    rows = (1 << 31) // 128
    slots = torch.arange(rows, device=DEV, dtype=torch.int64)
    sc = torch.full((1,), scale, dtype=torch.float32, device=DEV)
    first, code = _oracle_code_steps(scale)
    halves = []
    for start in (0, -(1 << 31)):               # patterns 0x00000000.., then 0x80000000..
        bits = torch.arange(start, start + (1 << 31), device=DEV, dtype=torch.int64).to(torch.int32)
        x = bits.view(torch.float32).view(rows, 1, 128)
        kc = torch.zeros((rows // 16, 1, 16, 128), dtype=torch.uint8, device=DEV)
        vc = torch.zeros_like(kc)
        pkv.append(x, x, slots, kc, vc, sc, sc)
        torch.cuda.synchronize()
        assert torch.equal(kc, vc)
        del bits, x, vc
        halves.append(kc.view(-1))
    pos, neg = halves
    # positive finite patterns: the steps of the code sequence
    fin = pos[:n_fin]
    assert int(fin[0]) == 0
    at = (torch.nonzero(fin[1:] != fin[:-1]).view(-1) + 1)
    got_first = at.cpu().numpy()
    got_code = fin[at].cpu().numpy().astype(np.int64)
    assert np.array_equal(got_first, first)
    assert np.array_equal(got_code, code)
    assert torch.all((pos[n_fin:] & 0x7F) == 0x7F)     # NaN patterns
    # negative patterns: the magnitude's code with the sign bit
    assert torch.equal(neg[:n_fin], fin | 0x80)
    assert torch.all((neg[n_fin:] & 0x7F) == 0x7F)


# ------------------------------------------------------------------ decode


def test_tiny_workload_matches_oracle():
    case = W.make_case("tiny", device=DEV)
    S.poison_unused(case)
    snaps = snaps_for(case)
    out = S.run_step(case, 0)
    worst = check_all_units(case, out, 0, snaps)
    assert worst < 2e-3
    assert out.shape == (2, 4, 64)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("D,G,H_kv,bs", [(128, 8, 2, 16), (128, 8, 1, 32), (64, 4, 2, 16),
                                          (64, 16, 1, 32), (128, 1, 3, 16), (128, 16, 2, 16),
                                          (64, 3, 2, 32), (128, 6, 1, 16)])
def test_decode_sweep_matches_oracle(kv, D, G, H_kv, bs):
    case = small_case(kv=kv, D=D, G=G, H_kv=H_kv, bs=bs, B=4, ctx_range=(1, 700),
                      seed=1000 + D + G * 7 + bs)
    if kv == "e4m3":
        case["k_cache"].fill_(S.E4M3_NAN)
        case["v_cache"].fill_(S.E4M3_NAN)
        S.fill_fp8_cache(case)
    else:
        S.poison_unused(case)
    snaps = snaps_for(case)
    for st in (0, -1, 64, 256):
        # re-running rewrites the same slot with the same token
        out = S.run_step(case, 0, split_tokens=st)
        check_all_units(case, out, 0, snaps)


def test_ragged_lengths_around_tile_and_block_edges():
    ctx = [0, 14, 15, 16, 30, 31, 32, 63, 64, 65, 127, 128]       # before the append
    case = small_case(kv="bf16", D=128, G=8, H_kv=1, bs=32, B=len(ctx), ctx=ctx, seed=77)
    S.poison_unused(case)
    snaps = snaps_for(case)
    for st in (0, -1, 64):
        out = S.run_step(case, 0, split_tokens=st)
        check_all_units(case, out, 0, snaps)


def test_empty_context_gives_zero_rows():
    case = small_case(kv="bf16", D=64, G=4, H_kv=2, bs=16, B=3, ctx=[5, 9, 3], seed=5)
    dev = DEV
    bt = case["block_tables"].to(dev)
    lens = torch.tensor([0, 10, 0], dtype=torch.int32, device=dev)
    for st in (0, -1, 64):
        out = pkv.decode_attention(case["q"][0], case["k_cache"], case["v_cache"], bt, lens,
                                   case["scale"], max_context_len=10, split_tokens=st)
        o = out.cpu()
        assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
        assert torch.all(torch.isfinite(o[1])) and o[1].abs().sum() > 0


def test_split_count_does_not_change_the_result():
    case = small_case(kv="bf16", D=128, G=8, H_kv=2, bs=16, B=3, ctx=[3000, 1500, 4095], seed=9,
                      q_mult=4.0)
    outs = [S.run_step(case, 0, split_tokens=st).cpu() for st in (0, -1, 64, 256, 1024, 4096)]
    for o in outs[1:]:
        assert torch.max(torch.abs(o - outs[0])) < 1e-5


def test_balanced_split_with_empty_sequences_between_others():
    case = small_case(kv="bf16", D=128, G=8, H_kv=2, bs=16, B=6, ctx=[0, 0, 3000, 0, 17, 0], seed=61)
    S.poison_unused(case)
    snaps = snaps_for(case)
    dev = DEV
    bt = case["block_tables"].to(dev)
    lens = torch.tensor([0, 0, 3001, 0, 18, 0], dtype=torch.int32, device=dev)
    slots = pkv.slot_mapping(bt, torch.tensor([3000, 17], device=dev), case["k_cache"],
                             seq_index=torch.tensor([2, 4], device=dev))
    pkv.append(case["k_new"][0][[2, 4]].contiguous(), case["v_new"][0][[2, 4]].contiguous(), slots,
               case["k_cache"], case["v_cache"])
    out = pkv.decode_attention(case["q"][0], case["k_cache"], case["v_cache"], bt, lens, case["scale"],
                               max_context_len=3001, split_tokens=-1).cpu().numpy()
    G = 8
    for b in (0, 1, 3, 5):
        assert np.all(out[b] == 0)
    for b in (2, 4):
        for h in range(2):
            ref = S.oracle_unit(case, b, h, 0, snaps[(b, h)])
            assert np.max(np.abs(out[b, h * G:(h + 1) * G] - ref)) <= 2e-3


def test_one_long_sequence_cut_into_many_pieces():
    # 1 sequence x 1 KV head: every warp of the balanced split takes a piece
    case = small_case(kv="bf16", D=128, G=8, H_kv=1, bs=32, B=1, ctx=[40000], seed=62, q_mult=4.0)
    snaps = snaps_for(case)
    plan = pkv.decode_plan(1, 8, case["k_cache"], 40001, split_tokens=-1)
    assert plan.mode == 0
    out = S.run_step(case, 0, split_tokens=-1)
    check_all_units(case, out, 0, snaps)
    ref_fixed = S.run_step(case, 0, split_tokens=1024)
    assert torch.max(torch.abs(out - ref_fixed)) < 1e-5


def test_all_contexts_empty():
    case = small_case(kv="bf16", D=64, G=4, H_kv=2, bs=16, B=3, ctx=[4, 4, 4], seed=63)
    lens = torch.zeros(3, dtype=torch.int32, device=DEV)
    for st in (0, -1):
        out = pkv.decode_attention(case["q"][0], case["k_cache"], case["v_cache"],
                                   case["block_tables"].to(DEV), lens, case["scale"],
                                   max_context_len=0, split_tokens=st)
        assert torch.all(out == 0)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_batch_above_balanced_limit_uses_fixed_splits(kv):
    case = small_case(kv=kv, D=64, G=4, H_kv=1, bs=16, B=2100, ctx_range=(1, 80), seed=64)
    if kv == "e4m3":
        case["k_cache"].fill_(S.E4M3_NAN)
        case["v_cache"].fill_(S.E4M3_NAN)
        S.fill_fp8_cache(case)
    else:
        S.poison_unused(case)
    assert pkv.decode_plan(2100, 4, case["k_cache"], 81).mode == 1
    assert pkv.decode_plan(2100, 4, case["k_cache"], 81, split_tokens=-1).mode == 1
    units = [(b, 0) for b in (0, 1, 777, 2099)]
    snaps = snaps_for(case, units)
    out = S.run_step(case, 0).cpu().numpy()
    for b, h in units:
        ref = S.oracle_unit(case, b, h, 0, None if snaps is None else snaps[(b, h)])
        assert np.max(np.abs(out[b, 0:4] - ref)) <= S.tolerance(case)


def test_block_relabelling_gives_identical_output():
    case = small_case(kv="bf16", D=128, G=8, H_kv=2, bs=16, B=3, ctx_range=(100, 900), seed=21)
    out = S.run_step(case, 0).clone()
    nb = case["num_blocks"]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(4))
    kc2 = torch.empty_like(case["k_cache"])
    vc2 = torch.empty_like(case["v_cache"])
    kc2[perm.to(DEV)] = case["k_cache"]
    vc2[perm.to(DEV)] = case["v_cache"]
    bt = case["block_tables"]
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).to(torch.int64)].to(torch.int32), bt)
    lens = (case["ctx"] + 1).to(DEV)
    out2 = pkv.decode_attention(case["q"][0], kc2, vc2, bt2.to(DEV), lens, case["scale"],
                                max_context_len=int(lens.max()))
    assert torch.equal(out, out2)


def test_unused_table_entries_are_never_read():
    case = small_case(kv="bf16", D=64, G=4, H_kv=1, bs=16, B=2, ctx=[20, 40], seed=31)
    out = S.run_step(case, 0).clone()
    bt = case["block_tables"].clone()
    bt[bt < 0] = 2 ** 31 - 1
    lens = (case["ctx"] + 1).to(DEV)
    out2 = pkv.decode_attention(case["q"][0], case["k_cache"], case["v_cache"], bt.to(DEV), lens,
                                case["scale"], max_context_len=int(lens.max()))
    assert torch.equal(out, out2)
    assert pkv.device_error(DEV) == 0


def test_pooled_entry_point_matches_caller_workspace():
    case = small_case(kv="bf16", D=128, G=8, H_kv=2, bs=16, B=3, ctx=[5000, 700, 2500], seed=13)
    out = S.run_step(case, 0).clone()
    lens = (case["ctx"] + 1).to(DEV)
    out2 = torch.empty_like(out)
    pkv.decode_attention_pooled(case["q"][0], case["k_cache"], case["v_cache"],
                                case["block_tables"].to(DEV), lens, case["scale"], int(lens.max()), out2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_device_error_word_reports_bad_values_without_faulting():
    case = small_case(kv="bf16", D=128, G=8, H_kv=1, bs=16, B=2, ctx=[40, 40], seed=41)
    assert pkv.device_error(DEV) == 0
    bt = case["block_tables"].clone()
    bt[1, 1] = case["num_blocks"] + 5                # a used entry pointing past the pool
    lens = torch.tensor([41, 41], dtype=torch.int32, device=DEV)
    out = pkv.decode_attention(case["q"][0], case["k_cache"], case["v_cache"], bt.to(DEV), lens,
                               case["scale"], max_context_len=41)
    assert pkv.device_error(DEV) == 2
    assert torch.all(torch.isfinite(out))
    # a context length beyond the host bound is clamped and reported
    lens2 = torch.tensor([41, 47], dtype=torch.int32, device=DEV)
    pkv.decode_attention(case["q"][0], case["k_cache"], case["v_cache"], case["block_tables"].to(DEV),
                         lens2, case["scale"], max_context_len=41)
    assert pkv.device_error(DEV) == 3
    # an append slot past the cache is dropped and reported
    kn = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device=DEV)
    before = case["k_cache"].clone()
    pkv.append(kn, kn, torch.tensor([case["num_blocks"] * 16], device=DEV), case["k_cache"], case["v_cache"])
    assert pkv.device_error(DEV) == 4
    assert torch.equal(before, case["k_cache"])
    assert pkv.device_error(DEV) == 0


# ------------------------------------------------------------ full-size workloads
# Every (sequence, KV head) unit of each workload is compared with the oracle,
# which runs on the host cores in a spawn pool (tests/oracle_pool.py) from the
# generator's inputs taken before the GPU touched the caches.


def _all_units(case):
    return [(b, h) for b in range(case["B"]) for h in range(case["H_kv"])]


@pytest.mark.parametrize("name,units", [("gqa_bf16", 512), ("shared_prefix", 1024)])
def test_full_size_bf16_workloads_every_unit(name, units):
    case = W.make_case(name, device=DEV)
    src = OP.UnitSource(case)
    out = S.run_step(case, 0).cpu().numpy()
    assert pkv.device_error(DEV) == 0
    assert np.all(np.isfinite(out))
    res = OP.run_units(src, _all_units(case), 1, [0])
    assert res["units"] == units
    assert OP.max_abs_err(out, res["outputs"], case["H_q"] // case["H_kv"]) <= 2e-3


def test_full_size_fp8_workload_fill_bit_exact_and_decode_every_unit():
    """B=256, contexts U[2048, 4096], E4M3 cache written by pkv.append from
    fp32 rows with per-(sequence, KV head) scales: every code the GPU wrote
    (the fill and the step's new token, all 2048 units) equals the oracle's
    encoding, and every unit's decode is within 5e-3 of the oracle on the
    oracle's own cache."""
    case = W.make_case("fp8", device=DEV)
    src = OP.UnitSource(case)
    S.fill_fp8_cache(case)
    out = S.run_step(case, 0).cpu().numpy()
    assert pkv.device_error(DEV) == 0
    res = OP.run_units(src, _all_units(case), 1, [0], want_codes=True)
    assert res["units"] == 2048
    assert OP.max_abs_err(out, res["outputs"], case["H_q"] // case["H_kv"]) <= 5e-3
    bs, D, H = case["bs"], case["D"], case["H_kv"]
    compared = 0
    for b in range(case["B"]):
        n = case["blocks_needed"][b]
        tokens = int(case["ctx"][b]) + 1
        ids = case["block_tables"][b, :n].to(torch.int64).to(DEV)
        gk = S.bytes8(case["k_cache"][ids].permute(1, 0, 2, 3).reshape(H, n * bs, D)[:, :tokens])
        gv = S.bytes8(case["v_cache"][ids].permute(1, 0, 2, 3).reshape(H, n * bs, D)[:, :tokens])
        for h in range(H):
            wk, wv = res["codes"][(b, h)]
            assert np.array_equal(gk[h], wk) and np.array_equal(gv[h], wv), (b, h)
            compared += 1
    assert compared == 2048


def test_full_size_long_context_steps_every_unit():
    """B=8 sequences of 131,072 tokens, q drawn x4 (a sharp softmax), 32
    append + decode steps with the context growing by one: all 64 units at
    steps 0, 15 and 31."""
    case = W.make_case("long_ctx", device=DEV)
    src = OP.UnitSource(case)
    checked = {}
    for s in range(case["steps"]):
        out = S.run_step(case, s)
        if s in (0, 15, case["steps"] - 1):
            checked[s] = out.cpu().numpy()
    assert pkv.device_error(DEV) == 0
    G = case["H_q"] // case["H_kv"]
    for s, got in checked.items():
        res = OP.run_units(src, _all_units(case), s + 1, [s])
        assert res["units"] == 64
        assert OP.max_abs_err(got, res["outputs"], G) <= 2e-3, s


# ------------------------------------------------------------ slot mapping


def test_slot_mapping_matches_oracle_addressing():
    """pkv_slot_mapping against the oracle's slot rule on random tables:
    every valid (sequence, position) pair bit-exact, padding gives -1 with no
    error, and a position past the table or a table entry outside the pool
    gives -1 and its error code."""
    g = torch.Generator().manual_seed(31337)
    nb, nseq, mb = 500, 7, 20
    for bs in (16, 32):
        table = torch.randperm(nb, generator=g)[:nseq * mb].reshape(nseq, mb).to(torch.int32)
        kc = torch.empty((nb, 1, bs, 64), dtype=torch.bfloat16, device=DEV)
        n = 4000
        seq = torch.randint(0, nseq, (n,), generator=g)
        pos = torch.randint(0, mb * bs, (n,), generator=g)
        pos[::97] = -1
        got = pkv.slot_mapping(table.to(DEV), pos.to(DEV), kc, seq_index=seq.to(DEV)).cpu().tolist()
        want = [PA.slot_of(table[s].numpy(), p, bs) if p >= 0 else -1 for s, p in zip(seq.tolist(), pos.tolist())]
        assert got == want
        pos1 = torch.randint(0, mb * bs, (nseq,), generator=g)
        got1 = pkv.slot_mapping(table.to(DEV), pos1.to(DEV), kc).cpu().tolist()
        assert got1 == [PA.slot_of(table[s].numpy(), int(pos1[s]), bs) for s in range(nseq)]
        assert pkv.device_error(DEV) == 0
    t = table.to(DEV)
    got = pkv.slot_mapping(t, torch.tensor([mb * bs, 3], device=DEV), kc, seq_index=torch.tensor([0, 9], device=DEV))
    assert got.cpu().tolist() == [-1, -1]
    assert pkv.device_error(DEV) == 3
    bad = table.clone()
    bad[1, 0] = nb + 5
    bad[2, 0] = -1
    got = pkv.slot_mapping(bad.to(DEV), torch.tensor([3, 5], device=DEV), kc,
                           seq_index=torch.tensor([1, 2], device=DEV))
    assert got.cpu().tolist() == [-1, -1]
    assert pkv.device_error(DEV) == 2


# ------------------------------------------------------------ shutdown


def test_calls_after_shutdown_set_the_library_up_again():
    """pkv_shutdown frees the library's pool and side stream and forgets the
    device addresses and kernel limits it looked up; the next calls set them
    up again and give the same results (the pool path, the cascade call with
    its side stream, a multi-token call with shared memory beyond the
    default limit)."""
    case = small_case(kv="bf16", D=128, G=8, H_kv=2, bs=16, B=4, ctx_range=(300, 2000), seed=77)
    bt = case["block_tables"].to(DEV)
    lens = (case["ctx"] + 1).to(DEV)
    mx = int(lens.max())
    q = case["q"][0].contiguous()

    def calls():
        out = torch.empty((4, 16, 128), dtype=torch.float32, device=DEV)
        pkv.decode_attention_pooled(q, case["k_cache"], case["v_cache"], bt, lens, case["scale"], mx, out)
        qm = case["q"][0].unsqueeze(1).repeat(1, 4, 1, 1).contiguous()          # [B, 4, H_q, D]
        om = pkv.multi_query_attention(qm, case["k_cache"], case["v_cache"], bt, lens, case["scale"], mx)
        torch.cuda.synchronize()
        return out.cpu(), om.cpu()

    a = calls()
    assert pkv.library().pkv_shutdown() == 0
    b = calls()
    assert pkv.device_error(DEV) == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
