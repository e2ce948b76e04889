"""The fused append + decode call (pkv_decode_attention_append) on the GPU:
against pkv_append followed by the decode call on a copy of the same caches
(the same bytes in both caches and the same output, bit for bit), against the
oracle, and with a bad table entry at the new position."""

import numpy as np
import pytest
import torch

import paged_kv_cache_222_gb300 as pkv
import workloads as W
from tests import gpu_support as S

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(kv, D, G, H_kv, bs, ctx, seed):
    spec = dict(B=len(ctx), H_q=G * H_kv, H_kv=H_kv, D=D, bs=bs, kv=kv, free_frac=0.25, steps=1, seed=seed,
                q_mult=1.0, ctx=tuple(ctx))
    case = W.make_case(spec, device=DEV)
    if kv == "e4m3":
        S.fill_fp8_cache(case)
    return case


def _raw(t):
    return t.view(torch.uint8) if t.element_size() == 1 else t.view(torch.int16)


def _both(case, src, split, lens=None):
    """(fused out, reference out, fused caches, reference caches)."""
    fp8 = case["kv"] == "e4m3"
    bt = case["block_tables"].to(DEV)
    if lens is None:
        lens = (case["ctx"].to(DEV) + 1).to(torch.int32)
    mx = max(int(lens.max()), 1)
    dt = torch.bfloat16 if src == "bf16" else torch.float32
    kn = case["k_new"][0].to(dt).contiguous()
    vn = case["v_new"][0].to(dt).contiguous()
    ks, vs = (case["k_scale"], case["v_scale"]) if fp8 else (None, None)
    q = case["q"][0].contiguous()
    kc_r, vc_r = case["k_cache"].clone(), case["v_cache"].clone()
    kc_f, vc_f = case["k_cache"].clone(), case["v_cache"].clone()
    pos = lens.to(torch.int64) - 1                       # -1 (padding) where nothing is appended
    slots = pkv.slot_mapping(bt, pos, kc_r)
    pkv.append(kn, vn, slots, kc_r, vc_r, ks, vs)
    ref = pkv.decode_attention(q, kc_r, vc_r, bt, lens, case["scale"], ks, vs, max_context_len=mx,
                               split_tokens=split)
    got = pkv.decode_attention(q, kc_f, vc_f, bt, lens, case["scale"], ks, vs, max_context_len=mx,
                               split_tokens=split, k_new=kn, v_new=vn)
    torch.cuda.synchronize()
    return got, ref, (kc_f, vc_f), (kc_r, vc_r)


@pytest.mark.parametrize("kv,src,D,G,H_kv,bs,ctx,split", [
    ("bf16", "bf16", 128, 8, 2, 16, [0, 15, 16, 300, 2048, 1], 0),
    ("bf16", "bf16", 128, 8, 2, 16, [0, 15, 16, 300, 2048, 1], 256),   # several splits per sequence
    ("bf16", "f32", 64, 4, 2, 32, [31, 32, 33, 700, 5], 64),           # f32 rows rounded into bf16
    ("bf16", "bf16", 128, 16, 1, 16, [100, 4000, 63], 0),              # G = 16
    ("e4m3", "f32", 128, 8, 2, 16, [15, 16, 300, 2048], 0),            # quantised with the scales
    ("e4m3", "bf16", 128, 8, 1, 32, [31, 200, 1000], 128),
    ("e4m3", "f32", 64, 8, 2, 16, [1, 64, 65, 900], 256),
])
def test_fused_append_equals_append_then_decode(kv, src, D, G, H_kv, bs, ctx, split):
    case = _case(kv, D, G, H_kv, bs, ctx, seed=1300 + D + bs + split + len(ctx))
    got, ref, fused, refc = _both(case, src, split)
    assert pkv.device_error(DEV) == 0
    for a, b in zip(fused, refc):
        assert torch.equal(_raw(a), _raw(b))               # every cache byte, the new rows included
    assert torch.equal(got, ref)                            # the same arithmetic on the same bytes
    assert torch.all(torch.isfinite(got))


def test_fused_append_matches_the_oracle():
    case = _case("bf16", 128, 8, 2, 16, [0, 15, 16, 300, 1500], seed=1401)
    S.poison_unused(case)
    snaps = {(b, h): S.snapshot_sequence(case, b, h) for b in range(case["B"]) for h in range(case["H_kv"])}
    got, _, _, _ = _both(case, "bf16", 0)
    G = case["H_q"] // case["H_kv"]
    out = got.cpu().numpy()
    for (b, h), snap in snaps.items():
        want = S.oracle_unit(case, b, h, 0, snap)
        assert np.max(np.abs(out[b, h * G:(h + 1) * G] - want)) <= 2e-3
    assert pkv.device_error(DEV) == 0


def test_fused_append_skips_empty_sequences_and_reports_bad_entries():
    case = _case("bf16", 128, 8, 1, 16, [40, 40, 40], seed=1402)
    lens = torch.tensor([41, 0, 41], dtype=torch.int32, device=DEV)   # sequence 1 appends nothing
    got, ref, fused, refc = _both(case, "bf16", 0, lens=lens)
    assert pkv.device_error(DEV) == 0
    for a, b in zip(fused, refc):
        assert torch.equal(_raw(a), _raw(b))
    assert torch.equal(got, ref)
    assert torch.all(got[1] == 0)
    # a table entry past the pool at the new position: nothing is written there,
    # the error word says why, and nothing faults
    bt = case["block_tables"].clone()
    bt[2, 40 // 16] = case["num_blocks"] + 7
    kc, vc = case["k_cache"].clone(), case["v_cache"].clone()
    before = (kc.clone(), vc.clone())
    kn = case["k_new"][0].contiguous()
    only2 = torch.tensor([0, 0, 41], dtype=torch.int32, device=DEV)   # only sequence 2 appends
    out = pkv.decode_attention(case["q"][0].contiguous(), kc, vc, bt.to(DEV), only2,
                               case["scale"], max_context_len=41, k_new=kn, v_new=kn)
    assert pkv.device_error(DEV) == 2
    assert torch.all(torch.isfinite(out))
    assert torch.equal(_raw(kc), _raw(before[0])) and torch.equal(_raw(vc), _raw(before[1]))
    assert pkv.device_error(DEV) == 0
