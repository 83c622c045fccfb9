"""Element and scale codecs of the block-scaled FP4 formats.

Formats (names as on "Lucifer-CUTLASS TP3 virtual-padding audit", section
"Packed W2 weight is wrong", and "Current Bug: CuTeDSLMoERunner", section
"Bug 5"). Definitions are from the public OCP 8-bit floating point
specification and OCP Microscaling Formats (MX) v1.0:

* E2M1: sign | exponent(2, bias 1) | mantissa(1). Magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.
* E4M3 (the "fn" variant): bias 7, no infinities. 0x7F and 0xFF are NaN,
  the maximum is 448, and subnormals are m/8 * 2^-6.
* E8M0: unsigned exponent, 2^(e-127). 0xFF is NaN.

Encoders are round-to-nearest with ties to the even code, saturating to the
largest finite magnitude ("satfinite"). They work by brute-force comparison
against the midpoints of the sorted representable values.
"""
from __future__ import annotations

import numpy as np


def e2m1_decode(code) -> np.ndarray:
    c = np.asarray(code, dtype=np.int64) & 0xF
    s = c >> 3
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return np.where(s == 1, -mag, mag)


def e4m3_decode(byte) -> np.ndarray:
    b = np.asarray(byte, dtype=np.int64) & 0xFF
    s = b >> 7
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e8m0_decode(byte) -> np.ndarray:
    b = np.asarray(byte, dtype=np.int64) & 0xFF
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


# Every code's value, from the bit-field decoders above: decoding a large array
# is then one table lookup per element (the same values, only faster).
E2M1_TABLE = e2m1_decode(np.arange(16))               # code 0..15 -> fp64
E4M3_TABLE = e4m3_decode(np.arange(256))              # byte -> fp64 (NaN at 0x7F, 0xFF)
E8M0_TABLE = e8m0_decode(np.arange(256))              # byte -> fp64 (NaN at 0xFF)

# sorted non-negative finite magnitudes; the index is the magnitude code
E2M1_MAGS = e2m1_decode(np.arange(8))                 # 0 .. 6
E4M3_MAGS = e4m3_decode(np.arange(127))               # 0 .. 448 (0x7F is NaN)
E2M1_MAX = 6.0
E4M3_MAX = 448.0


def _rne_index(mags: np.ndarray, a: np.ndarray) -> np.ndarray:
    """Index of the nearest entry of ascending ``mags`` to |a|, ties to the even index.

    ``a`` must be finite and non-negative and must not exceed ``mags[-1]``.
    Midpoints of consecutive entries are exact in fp64, and so is each
    comparison of an fp32 value with them.
    """
    mids = 0.5 * (mags[:-1] + mags[1:])
    k = np.searchsorted(mids, a, side="left")          # number of midpoints < a
    tie = (k < len(mids)) & (mids[np.minimum(k, len(mids) - 1)] == a)
    # on a tie the candidates are k and k+1: keep the even one
    return np.where(tie & (k % 2 == 1), k + 1, k)


def e2m1_encode(v) -> np.ndarray:
    """fp32 -> E2M1 code (0..15), RNE, satfinite, sign kept (-0 -> 0x8). NaN is rejected."""
    v = np.asarray(v, dtype=np.float32)
    if np.isnan(v).any():
        raise ValueError("e2m1_encode: NaN input")
    a = np.minimum(np.abs(v).astype(np.float64), E2M1_MAX)
    idx = _rne_index(E2M1_MAGS, a)
    sign = np.signbit(v).astype(np.int64)
    return (sign << 3 | idx).astype(np.uint8)


def e4m3_encode(v) -> np.ndarray:
    """fp32 -> E4M3 byte, RNE, satfinite (|v| > 448 -> 448). NaN is rejected."""
    v = np.asarray(v, dtype=np.float32)
    if np.isnan(v).any():
        raise ValueError("e4m3_encode: NaN input")
    a = np.minimum(np.abs(v).astype(np.float64), E4M3_MAX)
    idx = _rne_index(E4M3_MAGS, a)
    sign = np.signbit(v).astype(np.int64)
    return (sign << 7 | idx).astype(np.uint8)
