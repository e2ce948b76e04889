"""Pins for the oracle's number formats (CPU only).

The oracle's bf16 and E4M3 codecs are checked against (a) PyTorch's own bf16
and float8_e4m3fn conversions (an independent library routine), (b) values
fixed by the formats' definitions, and (c) structural invariants (round trips,
ties to even at every midpoint, saturation).
"""

import numpy as np
import pytest
import torch

from oracle import formats as F


def _f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def test_bf16_decode_matches_torch_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = F.bf16_bits_to_f64(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _f32_sweep(rng):
    """Every exponent and sign, mantissas covering all rounding cases of bf16."""
    sign = np.array([0, 1], dtype=np.uint32) << 31
    exps = np.arange(256, dtype=np.uint32) << 23
    top = np.arange(0, 128, 7, dtype=np.uint32) << 16            # kept mantissa bits
    low = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    grid = (sign[:, None, None, None] | exps[None, :, None, None]
            | top[None, None, :, None] | low[None, None, None, :]).ravel()
    rand = rng.integers(0, 1 << 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    return _f32(np.concatenate([grid, rand]))


def test_f32_to_bf16_matches_torch_rne():
    x = _f32_sweep(np.random.default_rng(1))
    ours = F.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN in, NaN out (payload not pinned)
    assert np.all(np.isnan(F.bf16_bits_to_f64(ours[nan])))


def test_f32_to_bf16_ties_to_even():
    # 1 + 2^-8 lies half-way between bf16 1.0 (0x3F80) and 1 + 2^-7 (0x3F81)
    assert F.f32_to_bf16_bits(np.float32(1 + 2 ** -8)) == 0x3F80
    # 1 + 3*2^-8 lies half-way between 0x3F81 and 0x3F82: the even code wins
    assert F.f32_to_bf16_bits(np.float32(1 + 3 * 2 ** -8)) == 0x3F82
    assert F.f32_to_bf16_bits(np.float32(-(1 + 3 * 2 ** -8))) == 0xBF82


def test_e4m3_table_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(F.E4M3_VALUES), nan)
    assert np.array_equal(F.E4M3_VALUES[~nan], ref[~nan])


def test_e4m3_definition_points():
    v = F.E4M3_VALUES
    assert v[0x7E] == 448.0                       # largest finite: 1.75 * 2^8
    assert v[0x01] == 2.0 ** -9                   # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9               # largest subnormal
    assert v[0x08] == 2.0 ** -6                   # smallest normal
    assert v[0x38] == 1.0                         # exponent field = bias
    assert v[0x30] == 0.5
    assert v[0xB8] == -1.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x00] == 0.0 and v[0x80] == 0.0 and np.signbit(v[0x80])
    assert np.sum(np.isnan(v)) == 2               # no infinities, two NaNs
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)               # codes ordered by magnitude


def test_e4m3_encode_round_trip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = F.e4m3_to_f64(codes).astype(np.float32)
    assert np.array_equal(F.e4m3_encode(vals), codes)


@pytest.mark.parametrize("enc_fn", [F.e4m3_encode, F.e4m3_encode_exhaustive])
def test_e4m3_encode_midpoints_tie_to_even(enc_fn):
    pos = F.E4M3_VALUES[:0x7F]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)   # exact in fp32
    enc = enc_fn(mids)
    lower = np.arange(0x7E, dtype=np.uint8)
    expect = np.where(lower % 2 == 0, lower, lower + 1).astype(np.uint8)
    assert np.array_equal(enc, expect)
    assert np.array_equal(enc_fn(-mids), expect | 0x80)
    # one fp32 ulp either side of a midpoint rounds to the nearer code
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    assert np.array_equal(enc_fn(up), lower + 1)
    assert np.array_equal(enc_fn(dn), lower)


@pytest.mark.parametrize("enc_fn", [F.e4m3_encode, F.e4m3_encode_exhaustive])
def test_e4m3_encode_saturation_and_specials(enc_fn):
    x = np.array([448, 449, 464, 480, 1e6, np.inf, -np.inf, -1e30, np.nan, 0.0, -0.0,
                  2.0 ** -10, 2.0 ** -10 * 1.0000001, -(2.0 ** -11)], dtype=np.float32)
    enc = enc_fn(x)
    assert list(enc[:8]) == [0x7E] * 6 + [0xFE, 0xFE]
    assert enc[8] == 0x7F
    assert enc[9] == 0x00 and enc[10] == 0x80
    assert enc[11] == 0x00            # exactly half of 2^-9: tie to even (zero)
    assert enc[12] == 0x01            # just above half: rounds up
    assert enc[13] == 0x80            # negative underflow keeps its sign


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32) * 100,
        rng.uniform(-448, 448, 200_000).astype(np.float32),
        (rng.standard_normal(50_000) * 2.0 ** -8).astype(np.float32),
    ])
    ours = F.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    inr = np.abs(x) <= 448
    assert inr.sum() > 400_000
    assert np.array_equal(ours[inr], ref[inr])


def test_f32_div_is_binary32():
    x = np.float32(1.0)
    s = np.float32(3.0)
    q = F.f32_div(x, s)
    assert q.dtype == np.float32
    # correctly rounded binary32 quotient: the nearest float32 to 1/3
    exact = 1.0 / 3.0
    cands = [np.nextafter(q, np.float32(0)), q, np.nextafter(q, np.float32(1))]
    assert min(cands, key=lambda c: abs(float(c) - exact)) == q


@pytest.mark.parametrize("code", [0x00, 0x01, 0x08, 0x38, 0x7E, 0x80, 0xFE])
def test_e4m3_encode_decode_consistency(code):
    v = np.float32(F.E4M3_VALUES[code])
    assert F.e4m3_encode(np.array([v]))[0] == code


def test_e4m3_bracketing_encoder_equals_exhaustive_encoder():
    """The encoder that compares only the two magnitudes bracketing |y| gives
    the code the all-127-magnitude brute force gives: random fp32 bit patterns
    over every exponent, values within a few ulps of every code and of every
    midpoint between neighbouring codes, both signs, zeros, infinities, NaN."""
    rng = np.random.default_rng(20260502)
    bits = rng.integers(0, 2 ** 32, 1_500_000, dtype=np.uint64).astype(np.uint32)
    pos = F.E4M3_VALUES[:0x7F].astype(np.float32)
    mids = ((F.E4M3_VALUES[:0x7E] + F.E4M3_VALUES[1:0x7F]) / 2).astype(np.float32)
    near = []
    for base in (pos, mids, np.float32([448.0, 464.0, 480.0])):
        v = base.copy()
        for _ in range(4):
            v = np.nextafter(v, np.float32(np.inf))
            near.append(v)
        v = base.copy()
        for _ in range(4):
            v = np.nextafter(v, np.float32(0))
            near.append(v)
        near.append(base)
    near = np.concatenate(near)
    x = np.concatenate([bits.view(np.float32), near, -near,
                        np.float32([0.0, -0.0, np.inf, -np.inf, np.nan, 1e38, -1e-45])])
    assert np.array_equal(F.e4m3_encode(x), F.e4m3_encode_exhaustive(x))
