"""GPU parity of the host tier: whole blocks moved between the device cache
and a page-locked host pool by the library's copy kernel (bit for bit), and a
serving loop that swaps a sequence out to the host, lets the freed device
blocks be reused, swaps it back and decodes it, against the oracle."""

import numpy as np
import pytest
import torch

import paged_kv_cache_222_gb300 as pkv
from oracle import paged_attention as PA
from oracle.block_manager import BlockManagerModel

from .gpu_support import bits16, bytes8

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _raw(t):
    return bits16(t) if t.dtype == torch.bfloat16 else bytes8(t)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_device_host_round_trip_is_bit_exact(kv):
    gen = torch.Generator().manual_seed(20260401)
    shape = (40, 8, 16, 128)
    if kv == "bf16":
        kc = torch.randn(shape, generator=gen).to(torch.bfloat16).to(DEV)
        vc = torch.randn(shape, generator=gen).to(torch.bfloat16).to(DEV)
    else:
        kc = torch.randint(0, 256, shape, generator=gen, dtype=torch.int32).to(torch.uint8).to(DEV)
        vc = torch.randint(0, 256, shape, generator=gen, dtype=torch.int32).to(torch.uint8).to(DEV)
    hk, hv = pkv.host_pool_like(kc, 16)
    hk.zero_()
    hv.zero_()
    src = [3, 17, 39, 0, 22]
    hdst = [15, 0, 7, 8, 1]
    k0, v0 = _raw(kc), _raw(vc)
    pkv.copy_blocks_between(kc, vc, hk, hv, src, hdst)
    torch.cuda.synchronize()
    for s, d in zip(src, hdst):
        assert np.array_equal(_raw(hk[d]), k0[s]) and np.array_equal(_raw(hv[d]), v0[s])
    ddst = [30, 31, 32, 33, 34]
    pkv.copy_blocks_between(hk, hv, kc, vc, hdst, ddst)
    assert pkv.device_error(DEV) == 0
    k1, v1 = _raw(kc), _raw(vc)
    for s, d in zip(src, ddst):
        assert np.array_equal(k1[d], k0[s]) and np.array_equal(v1[d], v0[s])
    untouched = [b for b in range(40) if b not in ddst]
    assert np.array_equal(k1[untouched], k0[untouched])


def test_out_of_pool_ids_are_skipped_and_recorded():
    kc = torch.zeros((8, 1, 16, 64), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    hk, hv = pkv.host_pool_like(kc, 4)
    hk.fill_(1.0)
    hv.fill_(1.0)
    pkv.copy_blocks_between(hk, hv, kc, vc, [0, 4, 1], [2, 3, 8])
    assert pkv.device_error(DEV) == 2
    got = kc.float().cpu()
    assert torch.all(got[2] == 1.0) and torch.all(got[3] == 0.0) and torch.all(got[[0, 1, 4, 5, 6, 7]] == 0.0)


def test_swap_out_reuse_swap_in_decode():
    nb, nh, hkv, G, d, bs = 48, 32, 2, 4, 128, 16
    hq = hkv * G
    gen = torch.Generator().manual_seed(20260402)
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    hk, hv = pkv.host_pool_like(kc, nh)
    hk.zero_()
    hv.zero_()
    okc, ovc = _raw(kc), _raw(vc)                       # oracle device pool
    ohk, ohv = okc[:nh].copy() * 0, ovc[:nh].copy() * 0   # oracle host pool (zeros)
    bm = pkv.BlockManager(nb, bs)
    bm.set_host_blocks(nh)
    model = BlockManagerModel(nb, bs, num_host_blocks=nh)
    scale = d ** -0.5

    def append(ids, n):
        nonlocal okc, ovc
        slots, cows = bm.append(ids, n)
        mslots, mcows = model.append(ids, n)
        assert slots.tolist() == mslots and not mcows
        k = torch.randn((len(slots), hkv, d), generator=gen).to(torch.bfloat16)
        v = torch.randn((len(slots), hkv, d), generator=gen).to(torch.bfloat16)
        pkv.append(k.to(DEV), v.to(DEV), torch.from_numpy(slots).to(DEV), kc, vc)
        okc, ovc = PA.append(bits16(k), bits16(v), PA.BF16, np.array(mslots), okc, ovc, PA.BF16)

    def decode(ids):
        tbl, lens = bm.block_tables(ids, 16)
        rows, mlens = model.block_tables(ids, 16)
        assert tbl.tolist() == rows
        q = torch.randn((len(ids), hq, d), generator=gen).to(torch.bfloat16)
        out = pkv.decode_attention(q.to(DEV), kc, vc, torch.from_numpy(tbl).to(DEV),
                                   torch.from_numpy(lens).to(DEV), scale, max_context_len=int(lens.max()))
        want = PA.decode_attention(bits16(q), okc, ovc, PA.BF16, np.array(rows), np.array(mlens), scale)
        assert pkv.device_error(DEV) == 0
        assert np.abs(out.cpu().numpy() - want).max() <= 2e-3

    for s in range(4):
        bm.add_sequence(s)
        model.add_sequence(s)
    append([0, 1, 2, 3], [100, 57, 130, 20])
    decode([0, 1, 2, 3])
    # preempt sequence 1: its blocks go to the host, the device blocks are freed
    pairs = bm.swap_out(1)
    assert [tuple(p) for p in pairs.tolist()] == model.swap_out(1)
    pkv.copy_blocks_between(kc, vc, hk, hv, pairs[:, 0], pairs[:, 1])
    for a, b in pairs.tolist():
        ohk[b], ohv[b] = okc[a], ovc[a]
    # the freed blocks are reused (and overwritten) by the others
    append([0, 2, 3], [40, 30, 60])
    decode([0, 2, 3])
    # bring it back into whatever device blocks are free now
    pairs = bm.swap_in(1)
    assert [tuple(p) for p in pairs.tolist()] == model.swap_in(1)
    pkv.copy_blocks_between(hk, hv, kc, vc, pairs[:, 0], pairs[:, 1])
    for a, b in pairs.tolist():
        okc[b], ovc[b] = ohk[a], ohv[a]
    append([0, 1, 2, 3], [1, 1, 1, 1])
    decode([0, 1, 2, 3])
    assert np.array_equal(_raw(kc), okc) and np.array_equal(_raw(vc), ovc)
