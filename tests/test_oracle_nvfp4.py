"""Pins of the oracle's NVFP4 quantiser, global-scale convention and scale swizzle."""
import json
import os

import numpy as np
import pytest

from oracle import codecs, nvfp4

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "runner_bug_history.json")))
F32 = np.float32


def test_global_scale_matches_printed_input_scale():
    g = GOLD["bug5_global_scale"]
    gs = nvfp4.global_scale(g["calibration_amax"])
    # the checkpoint's input_scale is the dequant direction 1/g = amax/2688 ~ 0.000286
    assert abs(1.0 / float(gs) - g["input_scale"]) / g["input_scale"] < 2e-3
    assert nvfp4.global_scale(0.0) == 1.0


def test_too_small_scale_saturates_block_scales_at_448():
    g = GOLD["bug5_global_scale"]
    gs_cal = nvfp4.global_scale(g["calibration_amax"])
    v = np.linspace(-g["runtime_amax"], g["runtime_amax"], 64, dtype=F32).reshape(1, 64)
    _, sf = nvfp4.quantize_rows(v, gs_cal)
    assert (codecs.e4m3_decode(sf) == g["saturated_block_scale"]).all()
    # the scale computed from the runtime amax does not saturate
    _, sf2 = nvfp4.quantize_rows(v, nvfp4.global_scale(g["runtime_amax"]))
    assert (codecs.e4m3_decode(sf2) <= 448).all() and (codecs.e4m3_decode(sf2) < 448).any()


def test_l2_scale_differs_from_l1_scale():
    g = GOLD["bug6_l2_scale"]
    r = float(nvfp4.global_scale(g["l1_amax"])) / float(nvfp4.global_scale(g["l2_amax"]))
    assert 30 <= r <= 40  # "30x too small"


def test_quantize_worked_blocks():
    # block A: amax 6, g = 1 -> s = 1 -> sf = 1.0 (0x38), inv = 1, codes are the E2M1 encodings
    a = np.array([6, 3, -0.25, 0.75, 1.25, -1.75, 2.5, 3.5, 5, -6, 0, -0.0, 0.1, -4, 1.5, 2], dtype=F32)
    # block B: amax 7 -> a/6 = 1.1666667 -> sf = 1.125 (0x39) -> inv = 1/1.125
    b = np.array([7, -7, 3.5] + [0] * 13, dtype=F32)
    # block C: all zero -> sf = 0, inv = 0, codes 0 (keeping the sign of -0)
    c = np.array([0.0] * 15 + [-0.0], dtype=F32)
    q, sf = nvfp4.quantize_rows(np.concatenate([a, b, c]).reshape(1, 48), F32(1.0))
    assert list(sf[0]) == [0x38, 0x39, 0x00]
    assert list(q[0, :16]) == [7, 5, 8, 2, 2, 12, 4, 6, 6, 15, 0, 8, 0, 14, 3, 4]
    inv_b = F32(1.0) / F32(1.125)
    assert q[0, 16] == 7 and q[0, 17] == 15                      # 7 * inv = 6.22 -> saturates to 6
    assert q[0, 18] == codecs.e2m1_encode(F32(3.5) * inv_b)       # 3.111 -> 3
    assert q[0, 18] == 5
    assert list(q[0, 32:]) == [0] * 15 + [8]
    d = nvfp4.dequantize(q, sf, 1.0)
    assert d[0, 16] == 6 * 1.125 and d[0, 18] == 3 * 1.125


def test_subnormal_block_scale():
    # amax 6 with g = 2^-8 -> s = 2^-8 = 2 * 2^-9 -> E4M3 subnormal 0x02
    v = np.zeros((1, 16), dtype=F32)
    v[0, 0] = 6.0
    q, sf = nvfp4.quantize_rows(v, F32(2.0**-8))
    assert sf[0, 0] == 0x02 and q[0, 0] == 7


def test_dequant_error_bound_random():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((64, 256)) * rng.uniform(0.01, 50, (64, 1))).astype(F32)
    gs = nvfp4.global_scale(np.abs(v).max())
    q, sf = nvfp4.quantize_rows(v, gs)
    d = nvfp4.dequantize(q, sf, gs)
    step = codecs.e4m3_decode(sf) / float(gs)                     # value of one E2M1 unit
    err = np.abs(d - v).reshape(64, 16, 16)
    # the largest E2M1 gap is 2 units (4 -> 6): error <= 1 unit, plus fp32 slack for the scale rounding
    assert (err <= step[:, :, None] * 1.0 * (1 + 1e-6) + 1e-30).all()
    # the block amax is reconstructed within the E4M3 scale rounding (relative 1/16)
    amax = np.abs(v).reshape(64, 16, 16).max(axis=2)
    amax_d = np.abs(d).reshape(64, 16, 16).max(axis=2)
    assert (np.abs(amax_d - amax) <= amax * 0.0625 + 1e-30).all()


def test_pack_low_nibble_first():
    q = np.array([[1, 2, 15, 0]], dtype=np.uint8)
    p = nvfp4.pack_codes(q)
    assert list(p[0]) == [0x21, 0x0F]
    assert (nvfp4.unpack_codes(p) == q).all()


def _swizzle_by_tiles(S):
    """The 128x4 tile layout built by reshapes: each 128-row x 4-column tile is
    four 32-row sub-blocks; output line i (16 bytes) is row i of sub-block 0,
    then row i of sub-block 1, and so on. Tiles are ordered column-tile fastest
    inside each 128-row block."""
    R, C = S.shape
    t = S.reshape(R // 128, 128, C // 4, 4).transpose(0, 2, 1, 3)      # [rb, cb, 128, 4]
    t = t.reshape(R // 128, C // 4, 4, 32, 4).transpose(0, 1, 3, 2, 4)  # [rb, cb, 32, sub, 4]
    return t.reshape(-1)


def test_swizzle_formula_matches_tile_construction():
    rng = np.random.default_rng(4)
    for R, C in [(128, 4), (256, 16), (384, 8)]:
        S = rng.integers(0, 256, (R, C)).astype(np.uint8)
        assert (nvfp4.swizzle(S) == _swizzle_by_tiles(S)).all()
        assert (nvfp4.unswizzle(nvfp4.swizzle(S), R, C) == S).all()


def test_per_expert_swizzle_equals_whole_buffer_when_starts_are_aligned():
    """'Bug 1' / 'Bug 11': the GEMM expects each expert's 128-row block swizzled on its own.

    With every expert starting on a 128-row boundary, swizzling the whole padded
    buffer gives exactly the concatenation of the per-expert swizzles.
    Unaligned starts do not.
    """
    rng = np.random.default_rng(5)
    C = 16
    counts = [100, 0, 300, 1]
    blocks = []
    for c in counts:
        P = (c + 127) // 128 * 128
        b = np.zeros((P, C), dtype=np.uint8)
        b[:c] = rng.integers(1, 256, (c, C))
        blocks.append(b)
    whole = nvfp4.swizzle(np.concatenate(blocks))
    per_expert = np.concatenate([nvfp4.swizzle(b) for b in blocks if len(b)])
    assert (whole == per_expert).all()
    # unaligned (unpadded) starts: pack rows back to back, pad only the end
    packed = np.concatenate([b[:c] for b, c in zip(blocks, counts)])
    packed = np.concatenate([packed, np.zeros((len(per_expert) // C - len(packed), C), dtype=np.uint8)])
    assert not (nvfp4.swizzle(packed) == per_expert).all()


def test_e4m3_saturation_threshold_is_the_midpoint_464():
    """block_scales' saturation threshold: above 464 E4M3 rounding would leave 448 (0x7E); at or below it the
    scale byte is an ordinary rounding to 448 or less. Checked against torch's float8_e4m3fn conversion, which
    rounds to nearest even (and overflows to NaN instead of saturating)."""
    torch = pytest.importorskip("torch")
    s = np.array([448.0, 450.0, 463.99997, 464.0, np.nextafter(np.float32(464.0), np.float32(1e9)), 470.0, 500.0],
                 dtype=np.float32)
    t = torch.from_numpy(s).to(torch.float8_e4m3fn).float().numpy()
    rounds_above = ~(t <= 448.0)                       # NaN (overflow) or a value above 448
    assert list(rounds_above) == list(s > nvfp4.E4M3_SATURATES_ABOVE)
    # and the scale the quantiser takes for such a block is the saturated 448 byte
    v = np.zeros((1, 16), np.float32)
    v[0, 0] = 6.0 * 470.0                              # s = 470 with g = 1
    assert nvfp4.block_scales(v, 1.0)[0, 0] == np.float32(470.0)
    assert nvfp4.quantize_rows(v, 1.0)[1][0, 0] == 0x7E
