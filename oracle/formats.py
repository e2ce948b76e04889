"""Number formats used by the paged KV cache, written from their definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

* bfloat16: the upper 16 bits of an IEEE-754 binary32 word.  Decoding is a
  shift; encoding from binary32 is round-to-nearest, ties-to-even.
* FP8 E4M3 (OCP 8-bit floating point, "E4M3" variant): 1 sign bit, 4 exponent
  bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; the
  largest finite magnitude is 1.75 * 2^8 = 448 and the smallest subnormal is
  2^-9.  [FN] FAQ "How much HBM memory does FP8 KV-cache quantization save?"
  names E4M3 with per-head scaling factors for KV blocks; the encoding itself
  is the OCP definition.

Encoders here pick the nearest code by exact float64 distance to decoded
candidate codes, so a reader can check them against the definition by eye
(the E4M3 one compares the two codes that bracket the value; an exhaustive
twin compares all 127 and checks it).
"""

import numpy as np

# --------------------------------------------------------------------------
# bfloat16
# --------------------------------------------------------------------------


def bf16_bits_to_f64(bits):
    """Exact value of bf16 words ``bits`` (uint16 array) as float64."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _f32_bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def f32_to_bf16_bits(x):
    """Round binary32 values to bf16, nearest with ties to even (brute force).

    For every input the two bf16 neighbours that bracket it (truncation and the
    next code away from zero) are decoded exactly and the nearer one is taken;
    on an exact tie the one with an even last mantissa bit wins.  Overflow past
    the largest finite bf16 by at least half an ulp goes to infinity, as IEEE
    round-to-nearest does.  NaN inputs give a quiet NaN of the same sign.
    """
    x = np.asarray(x, dtype=np.float32)
    u = _f32_bits(x).ravel()
    sign = (u >> np.uint32(31)).astype(np.uint16)
    mag = u & np.uint32(0x7FFFFFFF)
    lo = (mag >> np.uint32(16)).astype(np.uint32)          # truncated magnitude code
    hi = lo + np.uint32(1)                                 # next code up
    xv = (mag.view(np.float32)).astype(np.float64)         # |x| exactly

    def code_value(c):
        v = ((c << np.uint32(16)).view(np.float32)).astype(np.float64)
        # the code after the largest finite one is infinity; for rounding it
        # sits where the next binade would start (2^128)
        return np.where(c == np.uint32(0x7F80), 2.0 ** 128, v)

    dlo = xv - code_value(lo)
    dhi = code_value(hi) - xv
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((lo & np.uint32(1)) == 1))
    out = np.where(pick_hi, hi, lo).astype(np.uint32)
    out = np.where(mag == 0x7F800000, np.uint32(0x7F80), out)          # +-inf stays inf
    isnan = mag > 0x7F800000
    out = np.where(isnan, np.uint32(0x7FC0), out)
    out = out.astype(np.uint16) | (sign << np.uint16(15))
    return out.reshape(x.shape)


# --------------------------------------------------------------------------
# FP8 E4M3
# --------------------------------------------------------------------------

E4M3_MAX = 448.0
E4M3_NAN_CODE = 0x7F


def _e4m3_value(code):
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        mag = m * 2.0 ** (1 - 7 - 3)          # subnormal: 0.mmm * 2^(1-bias)
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


# Value of each of the 256 codes, float64 (NaN for 0x7F / 0xFF).
E4M3_VALUES = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)

# Non-negative finite codes 0x00..0x7E in increasing order of magnitude.
_E4M3_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_E4M3_POS_VALUES = E4M3_VALUES[:0x7F]


def e4m3_to_f64(codes):
    """Exact value of E4M3 codes (uint8 array) as float64."""
    return E4M3_VALUES[np.asarray(codes).astype(np.uint8)]


def e4m3_encode(y):
    """Encode binary32 values to E4M3 with round-to-nearest-even, saturating.

    The nearest of the 127 non-negative finite magnitudes to |y| is taken,
    distances measured exactly in float64; on a tie the code with an even last
    mantissa bit wins.  Only the two magnitudes that bracket |y| can be
    nearest (the magnitudes are sorted), so those two are compared.
    Magnitudes at or beyond 448, infinities included, saturate to 448 (code
    0x7E).  The sign is kept, so a negative value that rounds to zero gives
    0x80.  NaN gives 0x7F.  ``e4m3_encode_exhaustive`` measures the distance to
    every magnitude instead and gives the same codes.
    """
    y = np.asarray(y, dtype=np.float32)
    v = y.ravel()
    neg = np.signbit(v)
    a = np.abs(v.astype(np.float64))
    top = _E4M3_POS_CODES.size - 1
    hi = np.minimum(np.searchsorted(_E4M3_POS_VALUES, a, side="left"), top)   # first magnitude >= |y|
    lo = np.maximum(hi - 1, 0)                                                  # the one below it
    d_lo = np.abs(a - _E4M3_POS_VALUES[lo])
    d_hi = np.abs(_E4M3_POS_VALUES[hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((_E4M3_POS_CODES[hi] & 1) == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a >= E4M3_MAX, np.uint8(0x7E), code)                       # satfinite
    code = code | (neg.astype(np.uint8) << np.uint8(7))
    code = np.where(np.isnan(v), np.uint8(E4M3_NAN_CODE), code)
    return code.reshape(y.shape)


def e4m3_encode_exhaustive(y, chunk=1 << 16):
    """Brute-force E4M3 encoder: the distance from |y| to every one of the 127
    non-negative finite magnitudes is measured in float64 and the nearest code
    wins; on a tie the even code wins.  Saturation, sign and NaN as
    ``e4m3_encode``.  Slow (one row of 127 distances per value): it checks the
    bracketing encoder on sweeps."""
    y = np.asarray(y, dtype=np.float32)
    flat = y.ravel()
    out = np.empty(flat.shape, dtype=np.uint8)
    for s in range(0, flat.size, chunk):
        v = flat[s:s + chunk]
        neg = np.signbit(v)
        a = np.abs(v.astype(np.float64))
        dist = np.abs(a[:, None] - _E4M3_POS_VALUES[None, :])         # [n, 127]
        best = dist.min(axis=1, keepdims=True)
        cand = dist == best
        # among equally near codes prefer the even one, else the lowest
        even = cand & ((_E4M3_POS_CODES[None, :] & 1) == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        code = pick.astype(np.uint8)
        code = np.where(a >= E4M3_MAX, np.uint8(0x7E), code)           # satfinite
        code = code | (neg.astype(np.uint8) << np.uint8(7))
        code = np.where(np.isnan(v), np.uint8(E4M3_NAN_CODE), code)
        out[s:s + chunk] = code
    return out.reshape(y.shape)


def f32_div(x, s):
    """IEEE binary32 division x / s, correctly rounded (numpy float32)."""
    return (np.asarray(x, dtype=np.float32) / np.asarray(s, dtype=np.float32)).astype(np.float32)
