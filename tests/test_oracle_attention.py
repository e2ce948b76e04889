"""Pins for the oracle's paged decode attention and KV append (CPU only).

Each test pins the oracle to something other than itself:

* PyTorch's scaled_dot_product_attention in float64 on contiguous K/V (an
  independent library routine), with the paged pool built from the dense
  tensors by reshaping into blocks, not by the oracle's slot arithmetic;
* closed forms: one token gives its V row; q = 0, or identical keys, give the
  mean of V; constant V rows give that constant; two tokens give a sigmoid mix;
* invariances: relabelling physical blocks (pool and table together), and
  shared prefix blocks versus private copies, give bit-identical outputs;
  NaN in never-read slots and table entries changes nothing;
* append: written slots carry exactly the encoded rows, nothing else moves.
"""

import math

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import paged_attention as PA


def bf16_bits(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def paged_from_dense(dense, bs, n_pool, rng):
    """Split dense [B, H_kv, ctx_max, D] per sequence into bs-token blocks placed
    at random physical ids.  Built with reshape, not slot arithmetic."""
    B, H, T, D = dense.shape
    nblk = -(-T // bs)
    padded = np.zeros((B, H, nblk * bs, D), dtype=dense.dtype)
    padded[:, :, :T] = dense
    blocks = padded.reshape(B, H, nblk, bs, D).transpose(0, 2, 1, 3, 4)   # [B, nblk, H, bs, D]
    ids = rng.permutation(n_pool)[: B * nblk].reshape(B, nblk)
    pool = np.zeros((n_pool, H, bs, D), dtype=dense.dtype)
    pool[ids.ravel()] = blocks.reshape(B * nblk, H, bs, D)
    return pool, ids.astype(np.int32)


def sdpa_ref(q, K, V, scale, ctx):
    """torch SDPA, float64, per sequence, K/V repeated over the query group."""
    B, H_q, D = q.shape
    H_kv = K.shape[1]
    G = H_q // H_kv
    out = np.zeros((B, H_q, D))
    for b in range(B):
        qq = torch.from_numpy(q[b][:, None, :])                               # [H_q, 1, D]
        kk = torch.from_numpy(K[b, :, : ctx[b]]).repeat_interleave(G, dim=0)  # [H_q, ctx, D]
        vv = torch.from_numpy(V[b, :, : ctx[b]]).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale)
        out[b] = o[:, 0, :].numpy()
    return out


@pytest.mark.parametrize("B,H_q,H_kv,D,bs,ctx", [
    (2, 4, 1, 64, 16, (38, 101)),
    (3, 8, 2, 32, 32, (1, 33, 64)),
    (2, 16, 1, 16, 16, (16, 17)),
    (1, 6, 3, 8, 16, (5,)),
])
def test_decode_matches_sdpa_float64(B, H_q, H_kv, D, bs, ctx):
    rng = np.random.default_rng(B * 1000 + D)
    T = max(ctx)
    q = torch.randn(B, H_q, D, generator=torch.Generator().manual_seed(3))
    K = torch.randn(B, H_kv, T, D, generator=torch.Generator().manual_seed(4))
    V = torch.randn(B, H_kv, T, D, generator=torch.Generator().manual_seed(5))
    qb, Kb, Vb = bf16_bits(q), bf16_bits(K), bf16_bits(V)
    kpool, table = paged_from_dense(Kb, bs, 64, np.random.default_rng(7))
    vpool, table2 = paged_from_dense(Vb, bs, 64, np.random.default_rng(7))
    assert np.array_equal(table, table2)
    scale = 1.0 / math.sqrt(D)
    out = PA.decode_attention(qb, kpool, vpool, PA.BF16, table, np.array(ctx), scale)
    ref = sdpa_ref(F.bf16_bits_to_f64(qb), F.bf16_bits_to_f64(Kb), F.bf16_bits_to_f64(Vb), scale, ctx)
    assert np.max(np.abs(out - ref)) < 1e-12


def _tiny_pool(rng, H_kv=1, D=8, bs=4, n_pool=8):
    k = rng.standard_normal((n_pool, H_kv, bs, D)).astype(np.float32)
    v = rng.standard_normal((n_pool, H_kv, bs, D)).astype(np.float32)
    return F.f32_to_bf16_bits(k), F.f32_to_bf16_bits(v)


def test_single_token_returns_its_value_row():
    rng = np.random.default_rng(0)
    kc, vc = _tiny_pool(rng)
    q = F.f32_to_bf16_bits(rng.standard_normal((1, 3, 8)).astype(np.float32))
    table = np.array([[5, 2]], dtype=np.int32)
    out = PA.decode_attention(q, kc, vc, PA.BF16, table, np.array([1]), 0.3)
    expect = F.bf16_bits_to_f64(vc[5, 0, 0])
    assert np.array_equal(out[0], np.broadcast_to(expect, (3, 8)))


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(1)
    kc, vc = _tiny_pool(rng)
    q = np.zeros((1, 2, 8), dtype=np.uint16)
    table = np.array([[6, 1, 3]], dtype=np.int32)
    out = PA.decode_attention(q, kc, vc, PA.BF16, table, np.array([10]), 1.0)
    rows = np.concatenate([F.bf16_bits_to_f64(vc[6, 0]), F.bf16_bits_to_f64(vc[1, 0]),
                           F.bf16_bits_to_f64(vc[3, 0, :2])])
    assert np.allclose(out[0], rows.mean(axis=0), rtol=0, atol=1e-14)


def test_equal_keys_give_mean_and_constant_values_give_constant():
    rng = np.random.default_rng(2)
    kc, vc = _tiny_pool(rng)
    kc[:] = kc[0, 0, 0]                        # every key identical
    q = F.f32_to_bf16_bits(rng.standard_normal((1, 2, 8)).astype(np.float32) * 5)
    table = np.array([[4, 7]], dtype=np.int32)
    out = PA.decode_attention(q, kc, vc, PA.BF16, table, np.array([7]), 0.5)
    rows = np.concatenate([F.bf16_bits_to_f64(vc[4, 0]), F.bf16_bits_to_f64(vc[7, 0, :3])])
    assert np.allclose(out[0], rows.mean(axis=0), rtol=0, atol=1e-14)

    kc2, vc2 = _tiny_pool(np.random.default_rng(3))
    c = F.f32_to_bf16_bits(np.linspace(-2, 2, 8).astype(np.float32))
    vc2[:] = c
    out2 = PA.decode_attention(q, kc2, vc2, PA.BF16, table, np.array([8]), 0.5)
    assert np.allclose(out2[0], F.bf16_bits_to_f64(c)[None, :], rtol=0, atol=1e-14)


def test_two_tokens_sigmoid_mix():
    rng = np.random.default_rng(4)
    kc, vc = _tiny_pool(rng)
    q = F.f32_to_bf16_bits(rng.standard_normal((1, 1, 8)).astype(np.float32))
    table = np.array([[3]], dtype=np.int32)
    sc = 0.7
    out = PA.decode_attention(q, kc, vc, PA.BF16, table, np.array([2]), sc)
    qf = F.bf16_bits_to_f64(q[0, 0])
    k0, k1 = F.bf16_bits_to_f64(kc[3, 0, 0]), F.bf16_bits_to_f64(kc[3, 0, 1])
    v0, v1 = F.bf16_bits_to_f64(vc[3, 0, 0]), F.bf16_bits_to_f64(vc[3, 0, 1])
    w0 = 1.0 / (1.0 + math.exp(sc * float(qf @ k1) - sc * float(qf @ k0)))
    assert np.allclose(out[0, 0], w0 * v0 + (1 - w0) * v1, rtol=0, atol=1e-13)


def test_empty_context_gives_zeros():
    rng = np.random.default_rng(5)
    kc, vc = _tiny_pool(rng)
    q = F.f32_to_bf16_bits(rng.standard_normal((2, 2, 8)).astype(np.float32))
    table = np.array([[1, 2], [3, 4]], dtype=np.int32)
    out = PA.decode_attention(q, kc, vc, PA.BF16, table, np.array([0, 5]), 1.0)
    assert np.array_equal(out[0], np.zeros((2, 8)))
    assert np.all(np.isfinite(out[1]))


def test_gqa_head_mapping_is_contiguous_groups():
    """Query heads 0..G-1 read KV head 0, G..2G-1 read KV head 1."""
    rng = np.random.default_rng(6)
    H_kv, G, D, bs = 2, 3, 8, 4
    kc, vc = _tiny_pool(rng, H_kv=H_kv, D=D, bs=bs)
    vc[:, 0] = F.f32_to_bf16_bits(np.float32(1.0))   # every V row of head 0 is ones
    vc[:, 1] = F.f32_to_bf16_bits(np.float32(-2.0))  # every V row of head 1 is -2
    q = F.f32_to_bf16_bits(rng.standard_normal((1, H_kv * G, D)).astype(np.float32))
    out = PA.decode_attention(q, kc, vc, PA.BF16, np.array([[0, 5]]), np.array([6]), 0.4)
    assert np.allclose(out[0, :G], 1.0, atol=1e-14)
    assert np.allclose(out[0, G:], -2.0, atol=1e-14)


def test_block_relabelling_is_bit_identical():
    rng = np.random.default_rng(8)
    kc, vc = _tiny_pool(rng, H_kv=2, D=8, bs=4, n_pool=16)
    q = F.f32_to_bf16_bits(rng.standard_normal((2, 4, 8)).astype(np.float32))
    table = np.array([[3, 9, 12, 0], [7, 1, 14, 2]], dtype=np.int32)
    ctx = np.array([15, 13])
    out = PA.decode_attention(q, kc, vc, PA.BF16, table, ctx, 0.35)
    perm = rng.permutation(16)                       # old id i -> new id perm[i]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    out2 = PA.decode_attention(q, kc2, vc2, PA.BF16, perm[table].astype(np.int32), ctx, 0.35)
    assert np.array_equal(out, out2)


def test_shared_prefix_blocks_equal_private_copies():
    rng = np.random.default_rng(9)
    kc, vc = _tiny_pool(rng, H_kv=1, D=8, bs=4, n_pool=16)
    q = F.f32_to_bf16_bits(rng.standard_normal((3, 2, 8)).astype(np.float32))
    # three sequences share physical blocks 4 and 11 (refcount 3) as tokens 0..7
    shared = np.array([[4, 11, 2], [4, 11, 6], [4, 11, 9]], dtype=np.int32)
    ctx = np.array([10, 12, 9])
    out_shared = PA.decode_attention(q, kc, vc, PA.BF16, shared, ctx, 0.5)
    # private copies: duplicate blocks 4 and 11 for sequences 1 and 2
    kc2, vc2 = kc.copy(), vc.copy()
    for src, dst in ((4, 13), (11, 14), (4, 15), (11, 0)):
        kc2[dst], vc2[dst] = kc[src], vc[src]
    private = np.array([[4, 11, 2], [13, 14, 6], [15, 0, 9]], dtype=np.int32)
    out_private = PA.decode_attention(q, kc2, vc2, PA.BF16, private, ctx, 0.5)
    assert np.array_equal(out_shared, out_private)


def test_unread_slots_and_table_entries_do_not_matter():
    rng = np.random.default_rng(10)
    kc, vc = _tiny_pool(rng, H_kv=1, D=8, bs=4, n_pool=8)
    q = F.f32_to_bf16_bits(rng.standard_normal((1, 2, 8)).astype(np.float32))
    table = np.array([[2, 5, 7, -1]], dtype=np.int32)
    ctx = np.array([9])                   # blocks 2, 5 full, token 0 of block 7
    out = PA.decode_attention(q, kc, vc, PA.BF16, table, ctx, 0.5)
    kc2, vc2 = kc.copy(), vc.copy()
    nan16 = np.uint16(0x7FC0)
    kc2[7, 0, 1:], vc2[7, 0, 1:] = nan16, nan16            # tail of the last block
    for blk in (0, 1, 3, 4, 6):                            # blocks nobody references
        kc2[blk], vc2[blk] = nan16, nan16
    table2 = table.copy()
    table2[0, 3] = 2 ** 31 - 1
    out2 = PA.decode_attention(q, kc2, vc2, PA.BF16, table2, ctx, 0.5)
    assert np.array_equal(out, out2)


def test_fp8_decode_matches_sdpa_on_dequantised_values():
    rng = np.random.default_rng(11)
    B, H_q, H_kv, D, bs = 2, 4, 2, 16, 16
    ctx = (20, 45)
    T = max(ctx)
    K = rng.standard_normal((B, H_kv, T, D)).astype(np.float32)
    V = rng.standard_normal((B, H_kv, T, D)).astype(np.float32)
    ks = (np.abs(K).max(axis=(2, 3)) / np.float32(448)).astype(np.float32)
    vs = (np.abs(V).max(axis=(2, 3)) / np.float32(448)).astype(np.float32)
    # codes through torch's float8 conversion (library), decoded by torch too
    kq = torch.from_numpy(K / ks[:, :, None, None]).to(torch.float8_e4m3fn)
    vq = torch.from_numpy(V / vs[:, :, None, None]).to(torch.float8_e4m3fn)
    kcodes = kq.view(torch.uint8).numpy()
    vcodes = vq.view(torch.uint8).numpy()
    kpool, table = paged_from_dense(kcodes, bs, 16, np.random.default_rng(12))
    vpool, _ = paged_from_dense(vcodes, bs, 16, np.random.default_rng(12))
    q = F.f32_to_bf16_bits(rng.standard_normal((B, H_q, D)).astype(np.float32))
    scale = 1.0 / math.sqrt(D)
    out = PA.decode_attention(q, kpool, vpool, PA.E4M3, table, np.array(ctx), scale, ks, vs)
    Kd = kq.to(torch.float64).numpy() * ks[:, :, None, None].astype(np.float64)
    Vd = vq.to(torch.float64).numpy() * vs[:, :, None, None].astype(np.float64)
    ref = sdpa_ref(F.bf16_bits_to_f64(q), Kd, Vd, scale, ctx)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_units_subset_matches_full():
    rng = np.random.default_rng(13)
    kc, vc = _tiny_pool(rng, H_kv=2, D=8, bs=4, n_pool=16)
    q = F.f32_to_bf16_bits(rng.standard_normal((2, 4, 8)).astype(np.float32))
    table = np.array([[3, 9, 12, 0], [7, 1, 14, 2]], dtype=np.int32)
    ctx = np.array([15, 13])
    full = PA.decode_attention(q, kc, vc, PA.BF16, table, ctx, 0.35)
    part = PA.decode_attention(q, kc, vc, PA.BF16, table, ctx, 0.35, units=[(1, 0)])
    assert np.array_equal(part[1, 0:2], full[1, 0:2])
    assert np.all(np.isnan(part[0]))


# ---------------------------------------------------------------- append


def test_append_bf16_copies_bits_and_touches_nothing_else():
    rng = np.random.default_rng(20)
    kc, vc = _tiny_pool(rng, H_kv=2, D=8, bs=4, n_pool=8)
    new_k = F.f32_to_bf16_bits(rng.standard_normal((3, 2, 8)).astype(np.float32))
    new_v = F.f32_to_bf16_bits(rng.standard_normal((3, 2, 8)).astype(np.float32))
    slots = np.array([5 * 4 + 3, -1, 0 * 4 + 1])
    k2, v2 = PA.append(new_k, new_v, PA.BF16, slots, kc, vc, PA.BF16)
    assert np.array_equal(k2[5, :, 3], new_k[0]) and np.array_equal(v2[5, :, 3], new_v[0])
    assert np.array_equal(k2[0, :, 1], new_k[2]) and np.array_equal(v2[0, :, 1], new_v[2])
    mask = np.ones(kc.shape[:3], dtype=bool)
    mask[5, :, 3] = False
    mask[0, :, 1] = False
    assert np.array_equal(k2[mask], kc[mask]) and np.array_equal(v2[mask], vc[mask])


def test_append_f32_to_e4m3_matches_torch_quantisation():
    rng = np.random.default_rng(21)
    N, H, D, bs, nb = 40, 2, 16, 16, 8
    x = (rng.standard_normal((N, H, D)) * 3).astype(np.float32)
    y = (rng.standard_normal((N, H, D)) * 3).astype(np.float32)
    ks = rng.uniform(0.01, 0.05, (N, H)).astype(np.float32)
    vs = rng.uniform(0.01, 0.05, (N, H)).astype(np.float32)
    slots = rng.permutation(nb * bs)[:N]
    kc = np.zeros((nb, H, bs, D), dtype=np.uint8)
    vc = np.zeros((nb, H, bs, D), dtype=np.uint8)
    k2, v2 = PA.append(x, y, PA.F32, slots, kc, vc, PA.E4M3, ks, vs, scale_row_stride=H)
    kq = torch.from_numpy(x / ks[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    inr = np.abs(x / ks[:, :, None]) <= 448
    got = k2[slots // bs, :, slots % bs]                    # [N, H, D]
    assert np.array_equal(got[inr], kq[inr])
    assert np.all(got[~inr] & 0x7F == 0x7E)                 # saturated
    assert got.shape == (N, H, D)
    assert np.array_equal(v2[slots // bs, :, slots % bs],
                          F.e4m3_encode(F.f32_div(y, vs[:, :, None])))


def test_append_per_head_broadcast_scale():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((3, 2, 8)).astype(np.float32)
    hs = np.array([0.01, 0.02], dtype=np.float32)
    kc = np.zeros((4, 2, 4, 8), dtype=np.uint8)
    k2, _ = PA.append(x, x, PA.F32, np.array([1, 6, 11]), kc, kc, PA.E4M3, hs, hs, scale_row_stride=0)
    for i, s in enumerate([1, 6, 11]):
        for h in range(2):
            expect = torch.from_numpy(x[i, h] / hs[h]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(k2[s // 4, h, s % 4], expect)


def test_append_then_decode_matches_dense_with_new_token():
    """Append of the new token followed by decode over ctx + 1 tokens equals
    dense attention over [cached K; new k]."""
    rng = np.random.default_rng(23)
    D, bs, H_kv, H_q = 16, 16, 1, 4
    ctx = 37
    T = ctx + 1
    K = rng.standard_normal((1, H_kv, T, D)).astype(np.float32)
    V = rng.standard_normal((1, H_kv, T, D)).astype(np.float32)
    Kb, Vb = F.f32_to_bf16_bits(K), F.f32_to_bf16_bits(V)
    kpool, table = paged_from_dense(Kb, bs, 8, np.random.default_rng(24))
    vpool, _ = paged_from_dense(Vb, bs, 8, np.random.default_rng(24))
    # wipe the new token's slot, then append it back
    tail_blk = table[0, ctx // bs]
    kpool[tail_blk, :, ctx % bs] = 0x7FC0
    vpool[tail_blk, :, ctx % bs] = 0x7FC0
    slot = PA.slot_of(table[0], ctx, bs)
    k2, v2 = PA.append(Kb[:, :, ctx], Vb[:, :, ctx], PA.BF16, np.array([slot]), kpool, vpool, PA.BF16)
    q = F.f32_to_bf16_bits(rng.standard_normal((1, H_q, D)).astype(np.float32))
    out = PA.decode_attention(q, k2, v2, PA.BF16, table, np.array([T]), 0.25)
    ref = sdpa_ref(F.bf16_bits_to_f64(q), F.bf16_bits_to_f64(Kb), F.bf16_bits_to_f64(Vb), 0.25, [T])
    assert np.max(np.abs(out - ref)) < 1e-12
