"""Pins for the oracle's multi-token (causal) paged attention (CPU only):

* torch scaled_dot_product_attention in float64 with an explicit boolean mask
  built by torch.tril (an independent library routine and mask construction);
* q_len = 1 is decode attention, bit for bit;
* closed forms: a sequence holding only its q_len new tokens gives V[0] for
  its first query; queries before the start of the sequence give zeros.
"""

import math

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import paged_attention as PA

from .test_oracle_attention import bf16_bits, paged_from_dense


@pytest.mark.parametrize("B,QL,H_q,H_kv,D,bs,ctx", [
    (2, 4, 8, 2, 32, 16, (38, 101)),
    (3, 16, 4, 1, 16, 16, (16, 17, 70)),
    (1, 2, 16, 2, 64, 32, (33,)),
    (2, 7, 6, 3, 8, 16, (7, 40)),
])
def test_multi_query_matches_masked_sdpa_float64(B, QL, H_q, H_kv, D, bs, ctx):
    T = max(ctx)
    g = torch.Generator().manual_seed(11 + QL)
    q = torch.randn(B, QL, H_q, D, generator=g)
    K = torch.randn(B, H_kv, T, D, generator=g)
    V = torch.randn(B, H_kv, T, D, generator=g)
    qb, Kb, Vb = bf16_bits(q), bf16_bits(K), bf16_bits(V)
    kpool, table = paged_from_dense(Kb, bs, 64, np.random.default_rng(9))
    vpool, _ = paged_from_dense(Vb, bs, 64, np.random.default_rng(9))
    scale = 1.0 / math.sqrt(D)
    out = PA.multi_query_attention(qb, kpool, vpool, PA.BF16, table, np.array(ctx), scale)
    G = H_q // H_kv
    qf = torch.from_numpy(F.bf16_bits_to_f64(qb))
    Kf = torch.from_numpy(F.bf16_bits_to_f64(Kb))
    Vf = torch.from_numpy(F.bf16_bits_to_f64(Vb))
    for b in range(B):
        c = ctx[b]
        mask = torch.ones(QL, c, dtype=torch.bool).tril(diagonal=c - QL)     # query i sees t <= c-QL+i
        qq = qf[b].permute(1, 0, 2)                                        # [H_q, QL, D]
        kk = Kf[b, :, :c].repeat_interleave(G, dim=0)
        vv = Vf[b, :, :c].repeat_interleave(G, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
        assert np.max(np.abs(out[b] - ref.permute(1, 0, 2).numpy())) < 1e-12


def test_single_query_is_decode():
    rng = np.random.default_rng(2)
    kc = F.f32_to_bf16_bits(rng.standard_normal((12, 2, 16, 32)).astype(np.float32))
    vc = F.f32_to_bf16_bits(rng.standard_normal((12, 2, 16, 32)).astype(np.float32))
    q = F.f32_to_bf16_bits(rng.standard_normal((3, 1, 4, 32)).astype(np.float32))
    table = rng.permutation(12)[:12].reshape(3, 4).astype(np.int32)
    lens = np.array([1, 30, 64])
    a = PA.multi_query_attention(q, kc, vc, PA.BF16, table, lens, 0.2)
    d = PA.decode_attention(q[:, 0], kc, vc, PA.BF16, table, lens, 0.2)
    assert np.array_equal(a[:, 0], d)


def test_first_new_token_of_a_fresh_sequence_sees_only_itself():
    rng = np.random.default_rng(4)
    kc = F.f32_to_bf16_bits(rng.standard_normal((4, 1, 16, 8)).astype(np.float32))
    vc = F.f32_to_bf16_bits(rng.standard_normal((4, 1, 16, 8)).astype(np.float32))
    q = F.f32_to_bf16_bits(rng.standard_normal((1, 5, 2, 8)).astype(np.float32))
    table = np.array([[3, 1]], dtype=np.int32)
    out = PA.multi_query_attention(q, kc, vc, PA.BF16, table, np.array([5]), 0.3)
    v0 = F.bf16_bits_to_f64(vc[3, 0, 0])
    assert np.array_equal(out[0, 0, 0], v0) and np.array_equal(out[0, 0, 1], v0)


def test_queries_before_the_sequence_start_give_zeros():
    rng = np.random.default_rng(5)
    kc = F.f32_to_bf16_bits(rng.standard_normal((4, 1, 16, 8)).astype(np.float32))
    vc = kc.copy()
    q = F.f32_to_bf16_bits(rng.standard_normal((1, 6, 1, 8)).astype(np.float32))
    out = PA.multi_query_attention(q, kc, vc, PA.BF16, np.array([[0, 1]], dtype=np.int32),
                                   np.array([2]), 0.3)
    assert np.all(out[0, :4] == 0.0)                  # positions -4..-1
    assert np.array_equal(out[0, 4, 0], F.bf16_bits_to_f64(vc[0, 0, 0]))
