"""Pins of the oracle's element/scale codecs against closed forms, exact
rational brute force and torch's own fp8 casts."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import codecs

# OCP Microscaling v1.0, FP4 E2M1 element table (codes 0..7, then negated)
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_table():
    got = codecs.e2m1_decode(np.arange(16))
    want = E2M1_TABLE + [-v for v in E2M1_TABLE]
    assert list(got[:8]) == want[:8]
    assert list(got[8:]) == want[8:]
    assert np.signbit(got[8])  # code 0x8 is -0


def test_e4m3_decode_matches_torch():
    raw = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = raw.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = codecs.e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert (got[~nan] == ref[~nan]).all()
    assert got[0x7E] == 448.0 and got[0x01] == 2.0**-9 and got[0x08] == 2.0**-6 and got[0x38] == 1.0


def test_e8m0_decode_closed_form():
    got = codecs.e8m0_decode(np.arange(256))
    for b in range(255):
        assert got[b] == float(Fraction(2) ** (b - 127))
    assert np.isnan(got[255])
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        ok = ~np.isnan(ref)
        assert (got[ok] == ref[ok]).all()


def _exact_rne(v: float, mags: list[float], maxv: float) -> int:
    """Exact rational nearest-magnitude index with ties to the even index."""
    a = min(abs(Fraction(v)), Fraction(maxv))
    best = None
    for i, m in enumerate(mags):
        d = abs(a - Fraction(m))
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def _probe_values(mags):
    """Every representable value, every midpoint and +-1 ulp around each, in fp32."""
    vals = []
    m = np.array(mags, dtype=np.float64)
    pts = list(m) + list(0.5 * (m[:-1] + m[1:]))
    for p in pts:
        p32 = np.float32(p)
        vals += [p32, np.nextafter(p32, np.float32(np.inf)), np.nextafter(p32, np.float32(0))]
    vals += [np.float32(m[-1] * 1.5), np.float32(m[-1] * 100), np.float32(1e-30), np.float32(0)]
    v = np.array(vals, dtype=np.float32)
    return np.concatenate([v, -v])


def test_e2m1_encode_against_exact_brute_force():
    vals = _probe_values(E2M1_TABLE)
    rng = np.random.default_rng(0)
    vals = np.concatenate([vals, rng.uniform(-8, 8, 4000).astype(np.float32)])
    got = codecs.e2m1_encode(vals)
    for v, c in zip(vals, got):
        want = _exact_rne(float(v), E2M1_TABLE, 6.0) | (8 if np.signbit(v) else 0)
        assert c == want, (float(v), int(c), want)


def test_e2m1_encode_ties_and_saturation():
    enc = lambda x: int(codecs.e2m1_encode(np.float32(x)))
    assert enc(0.25) == 0 and enc(0.75) == 2 and enc(1.25) == 2 and enc(1.75) == 4
    assert enc(2.5) == 4 and enc(3.5) == 6 and enc(5.0) == 6
    assert enc(7.0) == 7 and enc(1e9) == 7 and enc(-1e9) == 15
    assert enc(-0.0) == 8 and enc(-0.1) == 8 and enc(0.0) == 0


def test_e4m3_encode_against_exact_brute_force():
    mags = list(codecs.E4M3_MAGS)
    vals = _probe_values(mags)
    vals = vals[np.abs(vals) < 1e6]
    got = codecs.e4m3_encode(vals)
    for v, c in zip(vals, got):
        want = _exact_rne(float(v), mags, 448.0) | (0x80 if np.signbit(v) else 0)
        assert c == want, (float(v), int(c), want)


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.uniform(0, 448, 20000), np.exp(rng.uniform(-14, 6, 20000)),
        0.5 * (codecs.E4M3_MAGS[:-1] + codecs.E4M3_MAGS[1:]),
    ]).astype(np.float32)
    v = v[v <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = codecs.e4m3_encode(v)
    assert (got == ref).all()


def test_e4m3_saturates():
    assert int(codecs.e4m3_encode(np.float32(449.0))) == 0x7E
    assert int(codecs.e4m3_encode(np.float32(1e30))) == 0x7E
    assert int(codecs.e4m3_encode(np.float32(464.0))) == 0x7E   # midpoint to the (absent) 480
