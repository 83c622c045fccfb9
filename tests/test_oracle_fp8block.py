"""Pins of the oracle's block-FP8 codec and shared expert.

Each pin checks the oracle against something other than itself:
* the E4M3 code table itself (amax 448 gives scale 1, so every finite code
  must come back unchanged);
* scales that are powers of two, which make v / s exact;
* brute-force nearest-value search over all finite E4M3 values;
* the independence of 128-wide groups and 128 x 128 blocks on shapes that
  are not square, so a transposed block index fails;
* a textbook SwiGLU FFN on weights the codec represents exactly;
* the TP3 invariant of "Lucifer-CUTLASS TP3 virtual-padding audit": three
  shards of 768 (768, 768 and 512 real features of 2048) sum to the whole
  expert.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import codecs, fp8block, moe

F32 = np.float32
FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


def test_amax_448_gives_scale_one_and_returns_every_code():
    vals = codecs.e4m3_decode(FINITE).astype(F32)          # 254 values, amax 448
    v = np.zeros((1, 256), dtype=F32)
    v[0, :254] = vals
    v[0, 254:] = 448.0
    q, s = fp8block.quantize_groups(v)
    assert s.shape == (1, 2)
    assert s[0, 0] == 1.0 and s[0, 1] == 1.0
    assert (q[0, :254] == FINITE).all()
    assert (q[0, 254:] == 0x7E).all()


def test_power_of_two_scale_is_exact():
    rng = np.random.default_rng(3)
    codes = rng.choice(FINITE[(FINITE & 0x7F) <= 0x7E], size=(3, 384)).astype(np.uint8)
    for r in range(3):                                      # each group holds +-448 once, so amax = 448 * 2^e
        codes[r, ::128] = 0x7E
    exps = np.array([[-7, 0, 3], [-20, 5, -1], [2, 2, 2]])
    v = codecs.e4m3_decode(codes) * np.repeat(np.ldexp(1.0, exps), 128, axis=1)
    q, s = fp8block.quantize_groups(v.astype(F32))
    assert (s == np.ldexp(F32(1.0), exps)).all()
    # -0 is not produced by the generator's finite codes except 0x80, which decodes to -0 and must keep its sign
    assert (q == codes).all()


def test_rne_nearest_by_brute_force():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((4, 256)) * np.array([[1e-3], [1.0], [300.0], [1e4]])).astype(F32)
    q, s = fp8block.quantize_groups(v)
    grid = np.array(sorted(set(codecs.e4m3_decode(FINITE).tolist())))
    for t in range(4):
        for g in range(2):
            blk = v[t, g * 128:(g + 1) * 128]
            sc = s[t, g]
            assert sc == F32(F32(np.abs(blk).max()) / F32(448.0))
            for i in range(128):
                r = Fraction(float(F32(blk[i] / sc)))
                got = Fraction(float(codecs.e4m3_decode(q[t, g * 128 + i])))
                best = min(abs(r - Fraction(float(c))) for c in grid)
                assert abs(r - got) == best
                if abs(r) > 448:
                    assert abs(got) == 448


def test_zero_group_and_tiny_amax_give_zero_codes():
    v = np.zeros((2, 256), dtype=F32)
    v[1, 128] = np.float32(2.0 ** -149)                    # amax / 448 rounds to 0 in fp32
    q, s = fp8block.quantize_groups(v)
    assert (q == 0).all() and (s == 0).all()
    assert (fp8block.dequantize_groups(q, s) == 0).all()


def test_groups_are_independent():
    rng = np.random.default_rng(7)
    v = rng.standard_normal((5, 384)).astype(F32)
    q0, s0 = fp8block.quantize_groups(v)
    v2 = v.copy()
    v2[3, 200] = 1000.0                                     # group (3, 1)
    q1, s1 = fp8block.quantize_groups(v2)
    changed = s1 != s0
    assert changed[3, 1] and changed.sum() == 1
    diff = np.nonzero((q1 != q0).any(axis=1))[0]
    assert list(diff) == [3]
    assert (q1[3, :128] == q0[3, :128]).all() and (q1[3, 256:] == q0[3, 256:]).all()


def test_blocks_are_128_by_128_and_independent():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((256, 384)) * 0.02).astype(F32)
    q0, s0 = fp8block.quantize_blocks(w)
    assert s0.shape == (2, 3)
    for i in range(2):
        for j in range(3):
            assert s0[i, j] == F32(F32(np.abs(w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]).max()) / F32(448))
    w2 = w.copy()
    w2[130, 300] = 5.0                                      # block (1, 2)
    q1, s1 = fp8block.quantize_blocks(w2)
    assert (s1 != s0).sum() == 1 and s1[1, 2] != s0[1, 2]
    rows, cols = np.nonzero(q1 != q0)
    assert rows.min() >= 128 and cols.min() >= 256


def exact_weights(rng, R, K, exps):
    """A matrix whose 128 x 128 blocks the codec holds exactly: E4M3 values times 2^e, each block's amax 448 * 2^e."""
    codes = rng.choice(FINITE, size=(R, K)).astype(np.uint8)
    codes[::128, ::128] = 0x7E
    return (codecs.e4m3_decode(codes) * np.repeat(np.repeat(np.ldexp(1.0, exps), 128, 0), 128, 1)).astype(F32)


def test_shared_expert_equals_textbook_ffn_on_exact_weights():
    rng = np.random.default_rng(11)
    H, Is, n = 256, 384, 3
    w1 = exact_weights(rng, 2 * Is, H, rng.integers(-12, -8, size=(2 * Is // 128, H // 128)))
    w2 = exact_weights(rng, H, Is, rng.integers(-12, -8, size=(H // 128, Is // 128)))
    se = fp8block.quantize_shared(w1, w2)
    assert (fp8block.dequantize_blocks(se.w1_q, se.w1_s) == w1).all()
    x_bits = moe.f32_to_bf16_bits(rng.standard_normal((n, H)).astype(F32))
    got = fp8block.shared_out(x_bits, se, 1e30, quantize_activations=False)
    # textbook SwiGLU FFN, element by element: o_i = sum_f W2[i, f] * silu(g_f) * u_f
    x = moe.bf16_to_f64(x_bits)
    W1, W2 = w1.astype(np.float64), w2.astype(np.float64)
    for t in range(n):
        g = np.array([sum(W1[f, h] * x[t, h] for h in range(H)) for f in range(Is)])
        u = np.array([sum(W1[Is + f, h] * x[t, h] for h in range(H)) for f in range(Is)])
        a = g / (1.0 + np.exp(-g)) * u
        o = np.array([sum(W2[i, f] * a[f] for f in range(Is)) for i in range(H)])
        np.testing.assert_allclose(got[t], o, rtol=1e-10, atol=1e-12 * np.abs(o).max())


def test_clamp_applies_to_the_shared_expert():
    rng = np.random.default_rng(13)
    H, Is = 128, 128
    w1 = (rng.standard_normal((2 * Is, H)) * 0.5).astype(F32)
    w2 = (rng.standard_normal((H, Is)) * 0.05).astype(F32)
    se = fp8block.quantize_shared(w1, w2)
    x_bits = moe.f32_to_bf16_bits((rng.standard_normal((2, H)) * 4).astype(F32))
    a = fp8block.shared_out(x_bits, se, 10.0, quantize_activations=False)
    b = fp8block.shared_out(x_bits, se, 1e30, quantize_activations=False)
    assert not np.allclose(a, b)                           # some |gate| or |up| > 10 here


def test_tp3_shards_sum_to_the_whole_expert():
    rng = np.random.default_rng(17)
    H, I = 128, 2048
    w1 = (rng.standard_normal((2 * I, H)) * 0.02).astype(F32)
    w2 = (rng.standard_normal((H, I)) * 0.02).astype(F32)
    x_bits = moe.f32_to_bf16_bits(rng.standard_normal((2, H)).astype(F32))
    full = fp8block.shared_out(x_bits, fp8block.quantize_shared(w1, w2), 10.0)
    total = np.zeros_like(full)
    real = []
    for r in range(3):
        s1, s2 = fp8block.tp_shard(w1, w2, r, 3)
        assert s1.shape == (2 * 768, H) and s2.shape == (H, 768)
        real.append(int((np.abs(s2).sum(axis=0) > 0).sum()))
        total += fp8block.shared_out(x_bits, fp8block.quantize_shared(s1, s2), 10.0)
    assert real == [768, 768, 512]
    np.testing.assert_allclose(total, full, rtol=1e-12, atol=1e-12 * np.abs(full).max())


def test_shared_term_in_the_combine():
    rng = np.random.default_rng(19)
    n, H = 4, 128
    o = rng.standard_normal((n, H))
    ids = -np.ones((n, 2), dtype=np.int64)                  # no routed pair held: y is the shared output alone
    y = moe.moe_tokens(moe.f32_to_bf16_bits(np.zeros((n, H), F32)), ids, np.ones((n, 2)), None, F32(1), F32(1),
                       10.0, shared=o)
    assert (y == moe.f32_to_bf16_bits(o.astype(F32))).all()
