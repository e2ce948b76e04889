"""GPU parity of the copy-on-write block copy, and of a serving loop driven by
the native block manager (fork, copy-on-write, append, decode) against the
oracle: caches bit for bit, attention within the decode tolerance."""

import numpy as np
import pytest
import torch

import paged_kv_cache_222_gb300 as pkv
from oracle import paged_attention as PA
from oracle.block_manager import BlockManagerModel, copy_blocks as oracle_copy_blocks

from .gpu_support import bits16, bytes8

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _raw(t):
    return bits16(t) if t.dtype == torch.bfloat16 else bytes8(t)


def _random_cache(nb, hkv, bs, d, kv, gen):
    if kv == "bf16":
        w = torch.randint(-2**15, 2**15, (nb, hkv, bs, d), generator=gen, dtype=torch.int32)
        return w.to(torch.int16).view(torch.bfloat16).to(DEV)
    return torch.randint(0, 256, (nb, hkv, bs, d), generator=gen, dtype=torch.int32).to(torch.uint8).to(DEV)


@pytest.mark.parametrize("kv,d,bs,hkv,n_pairs", [
    ("bf16", 128, 16, 8, 1), ("bf16", 128, 32, 8, 300), ("bf16", 64, 16, 1, 7),
    ("e4m3", 128, 16, 8, 64), ("e4m3", 64, 32, 2, 5),
])
def test_copy_blocks_bit_exact(kv, d, bs, hkv, n_pairs):
    gen = torch.Generator().manual_seed(20260101 + n_pairs)
    nb = 2 * n_pairs + 8
    kc = _random_cache(nb, hkv, bs, d, kv, gen)
    vc = _random_cache(nb, hkv, bs, d, kv, gen)
    perm = torch.randperm(nb, generator=gen)
    src, dst = perm[:n_pairs], perm[n_pairs:2 * n_pairs]
    pairs = list(zip(src.tolist(), dst.tolist()))
    want_k = oracle_copy_blocks(_raw(kc), pairs)
    want_v = oracle_copy_blocks(_raw(vc), pairs)
    pkv.copy_blocks(kc, vc, src.to(torch.int32), dst.to(torch.int32))
    assert pkv.device_error(DEV) == 0
    assert np.array_equal(_raw(kc), want_k)
    assert np.array_equal(_raw(vc), want_v)


def test_copy_blocks_skips_and_records_bad_ids():
    gen = torch.Generator().manual_seed(20260102)
    kc = _random_cache(10, 2, 16, 64, "bf16", gen)
    vc = _random_cache(10, 2, 16, 64, "bf16", gen)
    before_k, before_v = _raw(kc), _raw(vc)
    pkv.copy_blocks(kc, vc, [1, 10, 2, -1], [5, 6, 7, 8])
    assert pkv.device_error(DEV) == 2                     # PKV_DEVERR_BLOCK_ID
    want_k = oracle_copy_blocks(before_k, [(1, 5), (2, 7)])
    want_v = oracle_copy_blocks(before_v, [(1, 5), (2, 7)])
    assert np.array_equal(_raw(kc), want_k) and np.array_equal(_raw(vc), want_v)
    assert pkv.device_error(DEV) == 0                     # read clears it


@pytest.mark.parametrize("kv,d,bs", [("bf16", 128, 16), ("bf16", 64, 32), ("e4m3", 128, 16)])
def test_serving_loop_with_fork_and_copy_on_write(kv, d, bs):
    """Prompt of one sequence, forked twice; decode steps append one token to
    every live sequence (the first of each forked block triggers a device
    copy), a sequence retires and a new one is admitted mid-way.  Every step:
    the native manager's slots and copies equal the model's, the device caches
    equal the oracle's caches bit for bit, and decode matches the oracle."""
    nb, hkv, G = 96, 2, 4
    hq = hkv * G
    gen = torch.Generator().manual_seed(20260103 + d + bs)
    fp8 = kv == "e4m3"
    src_dtype = torch.float32 if fp8 else torch.bfloat16
    cdtype = torch.uint8 if fp8 else torch.bfloat16
    kc = torch.zeros((nb, hkv, bs, d), dtype=cdtype, device=DEV)
    vc = torch.zeros_like(kc)
    okc, ovc = _raw(kc), _raw(vc)
    ks = (torch.rand(hkv, generator=gen) * 0.01 + 0.005) if fp8 else None
    vs = (torch.rand(hkv, generator=gen) * 0.01 + 0.005) if fp8 else None
    bm = pkv.BlockManager(nb, bs)
    model = BlockManagerModel(nb, bs)
    scale = d ** -0.5
    odt = PA.E4M3 if fp8 else PA.BF16

    def rows(n):
        x = torch.randn((n, hkv, d), generator=gen)
        return x if fp8 else x.to(torch.bfloat16)

    def oracle_rows(x):
        return x.numpy() if fp8 else bits16(x)

    def do_append(ids, n_new):
        nonlocal okc, ovc
        slots, cows = bm.append(ids, n_new)
        mslots, mcows = model.append(ids, n_new)
        assert slots.tolist() == mslots and [tuple(c) for c in cows.tolist()] == mcows
        if len(cows):
            pkv.copy_blocks(kc, vc, torch.from_numpy(cows[:, 0].copy()), torch.from_numpy(cows[:, 1].copy()))
            okc = oracle_copy_blocks(okc, mcows)
            ovc = oracle_copy_blocks(ovc, mcows)
        k_new, v_new = rows(len(slots)), rows(len(slots))
        pkv.append(k_new.to(DEV), v_new.to(DEV), torch.from_numpy(slots).to(DEV), kc, vc,
                   ks.to(DEV) if fp8 else None, vs.to(DEV) if fp8 else None,
                   scale_row_stride=0 if fp8 else None)
        okc, ovc = PA.append(oracle_rows(k_new), oracle_rows(v_new), PA.F32 if fp8 else PA.BF16,
                             np.array(mslots), okc, ovc, odt,
                             ks.numpy() if fp8 else None, vs.numpy() if fp8 else None, scale_row_stride=0)

    def decode_and_check(ids):
        mb = 16
        tbl, lens = bm.block_tables(ids, mb)
        rows_m, lens_m = model.block_tables(ids, mb)
        assert tbl.tolist() == rows_m and lens.tolist() == lens_m
        q = torch.randn((len(ids), hq, d), generator=gen).to(torch.bfloat16)
        kss = ks.repeat(len(ids), 1).contiguous() if fp8 else None
        vss = vs.repeat(len(ids), 1).contiguous() if fp8 else None
        out = pkv.decode_attention(q.to(DEV), kc, vc, torch.from_numpy(tbl).to(DEV),
                                   torch.from_numpy(lens).to(DEV), scale,
                                   kss.to(DEV) if fp8 else None, vss.to(DEV) if fp8 else None,
                                   max_context_len=int(lens.max()))
        assert pkv.device_error(DEV) == 0
        assert np.array_equal(_raw(kc), okc) and np.array_equal(_raw(vc), ovc)
        want = PA.decode_attention(bits16(q), okc, ovc, odt, np.array(rows_m), np.array(lens_m), scale,
                                   kss.numpy() if fp8 else None, vss.numpy() if fp8 else None)
        tol = 5e-3 if fp8 else 2e-3
        assert np.abs(out.cpu().numpy() - want).max() <= tol

    for m in (bm, model):
        m.add_sequence(0)
    do_append([0], [37])
    for child in (1, 2):
        bm.fork(0, child)
        model.fork(0, child)
    live = [0, 1, 2]
    for step in range(6):
        do_append(live, [1] * len(live))
        decode_and_check(live)
        if step == 2:
            bm.free_sequence(1)
            model.free_sequence(1)
            for m in (bm, model):
                m.add_sequence(3)
            do_append([3], [20])
            live = [0, 2, 3]
    assert bm.num_free() == model.num_free()
