"""Pins of the TP3 virtual-padding shard plan and the MXFP4 codec."""
import json
import os

import numpy as np
import pytest

from oracle import codecs, moe, mxfp4

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tp3_shard_plan.json")))


def test_tp3_plan_widths():
    m = GOLD["routed_moe"]
    p = mxfp4.tp_plan(m["original"], GOLD["tp"], m["align"], m["kernel_align"])
    assert p.logical_per_rank == m["logical_per_rank"] == 704
    assert p.virtual_global == m["virtual_global"] == 2112
    assert p.kernel_local == m["kernel_local"] == 768
    s = GOLD["shared_expert"]
    ps = mxfp4.tp_plan(s["original"], GOLD["tp"], s["align"], 128)
    assert (ps.logical_per_rank, ps.virtual_global) == (s["logical_per_rank"], s["virtual_global"])


def test_shard_offsets_and_tails_in_each_storage_unit():
    m = GOLD["routed_moe"]
    p = mxfp4.tp_plan(m["original"], 3, m["align"], m["kernel_align"])
    for key in ("w13_unpacked_rows", "w2_packed_bytes", "w2_e8m0_groups"):
        g = GOLD[key]
        for r in range(3):
            off, n, tail = mxfp4.shard_units(m["original"], p, r, g["unit"])
            assert off == g["source_offsets"][r], (key, r)
            assert off + n == g["source_ends"][r], (key, r)
            assert tail == g["zero_tail"][r], (key, r)
        if "unit_blind_wrong_offsets" in g:
            assert [mxfp4.shard_units(m["original"], p, r, g["unit"])[0] for r in range(3)] != g["unit_blind_wrong_offsets"]
            assert p.kernel_local // g["unit"] == g["kernel_axis"]


def test_monotonic_source_survives_shard_and_concat():
    m = GOLD["routed_moe"]
    p = mxfp4.tp_plan(m["original"], 3, m["align"], m["kernel_align"])
    for unit, width_units in [(1, 2048), (2, 1024), (32, 64)]:
        src = (np.arange(7 * width_units, dtype=np.int64) % 251 + 1).astype(np.uint8).reshape(7, width_units)
        parts = []
        for r in range(3):
            d = mxfp4.shard_axis(src, 1, m["original"], p, r, unit)
            off, n, tail = mxfp4.shard_units(m["original"], p, r, unit)
            assert d.shape[1] == p.kernel_local // unit
            assert (d[:, n:] == 0).all() and tail == d.shape[1] - n
            parts.append(d[:, :n])
        assert (np.concatenate(parts, axis=1) == src).all()


def test_mx_scale_is_floor_log2_amax_minus_2():
    v = np.zeros((4, 32), dtype=np.float32)
    v[0, 0] = 6.0        # floor(log2 6) = 2 -> X = 0 -> 6 is code 7
    v[1, 0] = 7.0        # X = 0 -> 7 saturates to 6
    v[2, 0] = 0.02       # floor(log2 0.02) = -6 -> X = -8
    v[2, 1] = -0.01
    q, s = mxfp4.mx_quantize_rows(v)
    assert list(s) == [127, 127, 127 - 8, 0]
    assert q[0, 0] == 7 and q[1, 0] == 7
    assert q[2, 0] == codecs.e2m1_encode(np.float32(0.02 * 256))  # 5.12 -> 6? nearest of {4, 6} is 6
    assert q[2, 0] == 7 and q[2, 1] == codecs.e2m1_encode(np.float32(-2.56))
    d = mxfp4.mx_dequantize(q, s)
    assert d[0, 0] == 6.0 and d[1, 0] == 6.0 and d[2, 0] == 6.0 / 256
    assert (d[3] == 0).all()


def _rand_w(rng, rows, cols, scale):
    return (rng.standard_normal((rows, cols)) * scale).astype(np.float32)


def test_tp3_partials_sum_to_the_full_width_layer():
    """The pin of "4. MoE hardware tests": TP3 shards summed equal the full-width layer (fp64 rounding only).
    A unit-blind W2 cut (byte offsets 0/384/768 for packed bytes) breaks it."""
    rng = np.random.default_rng(5)
    H, I, E, k, n = 64, 192, 3, 2, 5
    full = [(_rand_w(rng, 2 * I, H, 0.05), _rand_w(rng, H, I, 0.05)) for _ in range(E)]
    x_bits = moe.f32_to_bf16_bits(rng.standard_normal((n, H)).astype(np.float32))
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2], [1, 0]])
    p3 = mxfp4.tp_plan(I, 3, 32, 128)
    p1 = mxfp4.tp_plan(I, 1, 32, 128)
    assert (p3.logical_per_rank, p3.kernel_local, p1.kernel_local) == (64, 128, 256)
    ex1 = {e: mxfp4.mx_expert_shard(*full[e], p1, 0) for e in range(E)}
    ref = mxfp4.mx_moe_partials(x_bits, ids, lambda e: ex1[e], 10.0)
    tot = np.zeros_like(ref)
    for r in range(3):
        ex = {e: mxfp4.mx_expert_shard(*full[e], p3, r) for e in range(E)}
        tot += mxfp4.mx_moe_partials(x_bits, ids, lambda e: ex[e], 10.0)
    assert np.allclose(tot, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # the unit-blind W2 cut of "Packed W2 weight is wrong" (source offsets counted in kernel-width storage
    # units, rank * 128 columns here, instead of logical ones) does not sum to the layer
    def unit_blind(e, r):
        good = mxfp4.mx_expert_shard(*full[e], p3, r)
        q2, s2 = mxfp4.mx_quantize_rows(full[e][1])
        Ik = p3.kernel_local
        q = np.zeros((H, Ik), np.uint8)
        sc = np.zeros((H, Ik // 32), np.uint8)
        c = q2[:, r * Ik:(r + 1) * Ik]
        q[:, :c.shape[1]] = c
        sc[:, :c.shape[1] // 32] = s2[:, r * Ik // 32:r * Ik // 32 + c.shape[1] // 32]
        return good._replace(w2_q=q, w2_s=sc)
    bad = np.zeros_like(ref)
    for r in range(3):
        ex = {e: unit_blind(e, r) for e in range(E)}
        bad += mxfp4.mx_moe_partials(x_bits, ids, lambda e: ex[e], 10.0)
    assert not np.allclose(bad, ref, rtol=1e-3, atol=1e-6)


def test_layer_on_exactly_representable_weights_is_the_textbook_moe():
    """Weights built as E2M1 x 2^X per 32-block survive MX quantisation exactly, so the oracle's layer must
    equal a plain dense SwiGLU MoE on the original fp32 weights. That dense layer rounds h to bf16 through
    torch's own conversion."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    H, I, E, k, n, L = 64, 64, 2, 2, 4, 10.0
    vals = codecs.e2m1_decode(np.arange(16, dtype=np.uint8))

    def exact(rows, cols):
        q = rng.integers(0, 16, (rows, cols)).astype(np.uint8)
        q[:, ::32] = rng.choice([6, 7, 14, 15], size=(rows, cols // 32))  # |4| or |6|: amax sets X
        X = rng.integers(-9, -4, (rows, cols // 32))
        return (vals[q].reshape(rows, cols // 32, 32) * np.ldexp(1.0, X)[:, :, None]).reshape(rows, cols).astype(np.float32)

    full = [(exact(2 * I, H), exact(H, I)) for _ in range(E)]
    plan = mxfp4.tp_plan(I, 1, 32, 64)
    ex = {e: mxfp4.mx_expert_shard(*full[e], plan, 0) for e in range(E)}
    for e in range(E):
        assert np.array_equal(mxfp4.mx_dequantize(ex[e].w1_q, ex[e].w1_s), full[e][0].astype(np.float64))
    x_bits = moe.f32_to_bf16_bits(rng.standard_normal((n, H)).astype(np.float32))
    ids = np.array([[0, 1], [1, 0], [0, 1], [1, 0]])
    w = np.array([[0.7, 0.3], [0.6, 0.4], [0.5, 0.5], [0.9, 0.1]])
    got = mxfp4.mx_moe_tokens(x_bits, ids, w, lambda e: ex[e], L)
    xt = torch.from_numpy(sg_bf16_to_f32(x_bits)).double()
    y = torch.zeros(n, H, dtype=torch.float64)
    for t in range(n):
        for j in range(k):
            W1 = torch.from_numpy(full[ids[t, j]][0]).double()
            W2 = torch.from_numpy(full[ids[t, j]][1]).double()
            gu = W1 @ xt[t]
            g, u = gu[:I], gu[I:]
            h = torch.minimum(g, torch.tensor(L)) * torch.sigmoid(torch.minimum(g, torch.tensor(L))) * u.clamp(-L, L)
            h = h.float().bfloat16().double()
            y[t] += float(w[t, j]) * (W2 @ h).float().bfloat16().double()   # l2_out is BF16 ("Data Flow")
    ref = y.float().bfloat16().view(torch.int16).numpy().view(np.uint16)
    # the dense path rounds h and y exactly as the oracle does; only the fp64 summation order differs, which
    # cannot move a bf16 rounding here, so the bits must agree (a truncating or skipped h rounding would not)
    assert np.array_equal(got, ref)


def _torch_bf16(v64):
    import torch
    return torch.from_numpy(np.asarray(v64, dtype=np.float64)).float().bfloat16().double().numpy()


def test_bf16_round_is_round_to_nearest_even_through_fp32():
    """_bf16_round against torch's fp64 -> fp32 -> bf16 conversion, on exact bf16 ties (low half 0x8000 with
    even and odd high halves), the fp32 neighbours of every tie, exact bf16 values, and fp64 values a hair
    above or below a tie that fp32 rounding moves onto it."""
    pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    hi = rng.integers(0, 0x7F00, 2048).astype(np.uint32)            # finite, both parities of the last bf16 bit
    lows = np.array([0x8000, 0x7FFF, 0x8001, 0x0000, 0xFFFF, 0x4000, 0xC000], dtype=np.uint32)
    bits = ((hi[:, None] << 16) | lows[None, :]).reshape(-1)
    v32 = bits.view(np.float32).astype(np.float64)
    v = np.concatenate([v32, -v32, v32 * (1 + 2.0 ** -40), v32 * (1 - 2.0 ** -40), -v32 * (1 + 2.0 ** -40)])
    got = mxfp4._bf16_round(v)
    ref = _torch_bf16(v)
    assert np.array_equal(got.view(np.uint64), ref.view(np.uint64))
    # the ties themselves go to the even neighbour, which truncation (or no rounding) would not give
    tie = v32[(bits & 0xFFFF) == 0x8000]
    up = ((tie.astype(np.float32).view(np.uint32) >> 16) & 1) == 1
    r = mxfp4._bf16_round(tie).astype(np.float32).view(np.uint32) >> 16
    assert ((r & 1) == 0).all() and (r[up] == (tie[up].astype(np.float32).view(np.uint32) >> 16) + 1).all()


def test_expert_out_rounds_h_to_bf16_before_w2():
    """With W2 the identity (exact in MXFP4: 1 = E2M1 4 x 2^-2), mx_expert_out returns h itself after its bf16
    rounding. Checked bit for bit against torch's SwiGLU in fp64 rounded to bf16."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    H = I = 64
    vals = codecs.e2m1_decode(np.arange(16, dtype=np.uint8))
    q = rng.integers(0, 16, (2 * I, H)).astype(np.uint8)
    q[:, ::32] = 7                                                   # amax 6 per block: X = 0 after the shift
    w1 = (vals[q] * 2.0 ** -3).astype(np.float32)                    # exact in MXFP4
    w2 = np.eye(H, I, dtype=np.float32)
    ex = mxfp4.mx_expert_shard(w1, w2, mxfp4.tp_plan(I, 1, 32, 64), 0)
    assert np.array_equal(mxfp4.mx_dequantize(ex.w1_q, ex.w1_s), w1.astype(np.float64))
    assert np.array_equal(mxfp4.mx_dequantize(ex.w2_q, ex.w2_s), w2.astype(np.float64))
    x = sg_bf16_to_f32(moe.f32_to_bf16_bits((rng.standard_normal((16, H)) * 3).astype(np.float32))).astype(np.float64)
    o = mxfp4.mx_expert_out(ex, x, 10.0)
    gu = torch.from_numpy(x) @ torch.from_numpy(w1.astype(np.float64)).T      # exact: few-bit products, short sums
    g, u = gu[:, :I].clamp(max=10.0), gu[:, I:].clamp(-10.0, 10.0)
    h = (g * torch.sigmoid(g) * u).float().bfloat16().double().numpy()
    assert np.array_equal(o, h)
    assert not np.array_equal(o, (g * torch.sigmoid(g) * u).numpy())   # the rounding is really there


def sg_bf16_to_f32(u):
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------- MXFP4 weights in the NVFP4 operand form ----

def test_e4m3_powers_of_two():
    """Every power of two from 2^-9 to 2^8 has exactly one E4M3 byte, the one the codec decodes to it; the
    neighbours of the range have none (2^-10 underflows, 2^9 = 512 is past 448)."""
    from oracle import codecs
    for d in range(-9, 9):
        b = mxfp4.e4m3_pow2_byte(d)
        assert codecs.e4m3_decode(np.array([b], np.uint8))[0] == 2.0 ** d
        hits = [c for c in range(0x7F) if codecs.e4m3_decode(np.array([c], np.uint8))[0] == 2.0 ** d]
        assert hits == [b]
    for d in (-10, 9):
        with pytest.raises(ValueError):
            mxfp4.e4m3_pow2_byte(d)


def test_mx_as_nvfp4_is_exact_across_the_window():
    """Blocks spread over the whole 18-binade window, an all-zero block and a window-edge block: the NVFP4 form
    dequantises to the MX values bit for bit, and gw = 2^-(X_max - 8)."""
    from oracle import nvfp4
    rng = np.random.default_rng(5)
    v = rng.uniform(-1.0, 1.0, (128, 32, 32))
    v[:, :, 0] = 1.5                                   # every block's amax: 1.5 before its scaling
    exps = np.arange(32) % 18                          # block j scaled by 2^-(j % 18): X from -2 down to -19
    v = (v * np.ldexp(1.0, -exps)[None, :, None]).reshape(128, 1024).astype(np.float32)
    v[3, 64:96] = 0.0                                  # an all-zero block
    q, s = mxfp4.mx_quantize_rows(v)
    X = s.astype(int) - 127
    q2, sf, gw = mxfp4.mx_as_nvfp4(q, s)
    assert gw == np.float32(2.0 ** -(X[s > 0].max() - 8))
    assert np.array_equal(q2, q) and (sf[3, 4:6] == 0).all()
    assert np.array_equal(nvfp4.dequantize(q2, sf, gw), mxfp4.mx_dequantize(q, s))
    assert X[s > 0].max() - X[s > 0].min() == 17    # the window is full
    assert np.array_equal(sf[:, 0::2], sf[:, 1::2])     # both halves of a 32-element block share the scale


def test_mx_as_nvfp4_rejects_a_block_below_the_window():
    v = np.ones((128, 64), np.float32)
    v[0, 32:] = 2.0 ** -20                             # 20 binades below the rest
    q, s = mxfp4.mx_quantize_rows(v)
    with pytest.raises(ValueError):
        mxfp4.mx_as_nvfp4(q, s)
    s_nan = s.copy()
    s_nan[1, 0] = 0xFF
    with pytest.raises(ValueError):
        mxfp4.mx_as_nvfp4(q, s_nan)
