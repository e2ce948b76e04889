"""Pins for the footprint formula and the capacity arithmetic (CPU only).

Expected values are the ones the pages print, stored under tests/golden/ with
their citations.
"""

import os

import pytest

from oracle import footprint as FP

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _records(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def test_bytes_per_token_printed_values():
    n = 0
    for rec in _records("kv_footprint.txt"):
        if rec[0] == "bytes_per_token":
            L, nkv, d, p, expect = map(int, rec[1:])
            assert FP.kv_bytes_per_token(L, nkv, d, p) == expect
            n += 1
        elif rec[0] == "kib_per_token":
            L, nkv, d, p = map(int, rec[1:5])
            assert f"{FP.kv_bytes_per_token(L, nkv, d, p) / 1024:.1f}" == rec[5]
            n += 1
    assert n == 3


def test_size_table_printed_values_and_ratios():
    rows = [r for r in _records("kv_footprint.txt") if r[0] == "size_table"]
    assert len(rows) == 4
    sizes = []
    for _, S, B, p, printed, unit in rows:
        total = FP.kv_bytes(80, 8, 128, int(S), int(B), int(p))
        div = 1000 * 1024 ** (2 if unit == "GiB" else 3)
        assert f"{total / div:.2f}" == printed
        sizes.append(total)
    # ratios of the printed sizes are exact ratios of the formula
    assert sizes[1] == 16 * sizes[0]
    assert sizes[2] == 128 * sizes[0]
    assert sizes[3] == 1024 * sizes[0]


def test_footprint_is_linear_in_every_factor():
    base = FP.kv_bytes(2, 3, 5, 7, 11, 2)
    assert base == 2 * 2 * 3 * 5 * 7 * 11 * 2
    assert FP.kv_bytes(4, 3, 5, 7, 11, 2) == 2 * base
    assert FP.kv_bytes(2, 3, 5, 7, 22, 1) == base


def test_capacity_simulator_printed_output():
    golden = {(r[0], r[1]): r[2] for r in _records("capacity_simulator.txt")}
    common = dict(params_billion=70, n_layers=80, n_kv_heads=8, d_head=128, weight_bytes=2,
                  gpu_count=8, vram_per_gpu_gb=80, overhead_per_gpu_gb=3.5,
                  avg_ctx=1500, max_ctx=4096)
    r16 = FP.cluster_capacity(kv_bytes_per_elem=2, **common)
    r8 = FP.cluster_capacity(kv_bytes_per_elem=1, **common)
    assert f"{r16['kv_bytes_per_token'] / 1024:.1f}" == golden[("fp16", "kv_kib_per_token")]
    assert f"{r16['weights_gb']:.2f}" == golden[("fp16", "weights_gb")]
    assert f"{r16['weights_gb'] / 8:.1f}" == golden[("fp16", "weights_gb_per_gpu")]
    assert f"{r16['usable_kv_gb']:.1f}" == golden[("fp16", "usable_kv_gb")]
    assert str(r16["streams_contiguous"]) == golden[("fp16", "streams_contiguous")]
    assert str(r16["streams_paged"]) == golden[("fp16", "streams_paged")]
    assert str(r16["gain_percent"]) == golden[("fp16", "gain_percent")]
    assert f"{r8['kv_bytes_per_token'] / 1024:.1f}" == golden[("fp8", "kv_kib_per_token")]
    assert str(r8["streams_paged"]) == golden[("fp8", "streams_paged")]


@pytest.mark.parametrize("dtype_bytes", [1, 2])
def test_pool_bytes_per_token_for_one_layer(dtype_bytes):
    """For one layer the bytes a paged pool holds per cached token are
    2 * H_kv * D * p: the cache tensors [NB, H_kv, bs, D] for K and for V."""
    H_kv, D, bs, nb = 8, 128, 16, 10
    pool_bytes = 2 * nb * H_kv * bs * D * dtype_bytes
    assert pool_bytes // (nb * bs) == FP.kv_bytes_per_token(1, H_kv, D, dtype_bytes)
