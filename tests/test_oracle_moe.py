"""Pins of the oracle's router, softmax top-k, clamped SwiGLU and whole layer."""
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synthgen as sg
from oracle import layout, moe, nvfp4


def test_router_logits_are_the_exact_sum_rounded_once():
    rng = np.random.default_rng(0)
    x = sg.f32_to_bf16_bits(rng.standard_normal((3, 64)).astype(np.float32))
    w = sg.f32_to_bf16_bits(rng.standard_normal((5, 64)).astype(np.float32))
    l = moe.router_logits(x, w)
    xf, wf = sg.bf16_bits_to_f32(x), sg.bf16_bits_to_f32(w)
    for t in range(3):
        for e in range(5):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xf[t], wf[e]))
            assert l[t, e] == np.float32(float(exact))


def test_topk_matches_torch_topk_and_softmax():
    rng = np.random.default_rng(1)
    l = rng.standard_normal((50, 256)).astype(np.float32)
    ids, w = moe.topk_softmax(l, 6)
    tv, ti = torch.topk(torch.from_numpy(l).double(), 6, dim=1)
    assert (ids == ti.numpy()).all()
    ref = torch.softmax(tv, dim=1).numpy()
    assert np.allclose(w, ref, rtol=1e-13, atol=0)
    assert np.allclose(w.sum(1), 1.0, rtol=1e-14)
    # renormalised top-k equals the full softmax restricted to the selection
    full = torch.softmax(torch.from_numpy(l).double(), dim=1).numpy()
    sel = np.take_along_axis(full, ids, 1)
    assert np.allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-12)


def test_topk_ties_go_to_lower_expert():
    l = np.zeros((1, 8), dtype=np.float32)
    l[0, [2, 5, 7]] = 1.0
    ids, w = moe.topk_softmax(l, 4)
    assert list(ids[0]) == [2, 5, 7, 0]
    l[0, :] = -0.0
    l[0, 3] = 0.0
    ids, _ = moe.topk_softmax(l, 2)
    assert list(ids[0]) == [0, 1]  # -0 == +0


def test_topk_ranks_nan_below_every_number():
    """Brute force on small rows of numbers, +-0, +-inf and NaN: the k picks are the first k of the order
    (NaN after every number, -inf included; then value descending; then the lower id), so a NaN logit is
    picked only when fewer than k numbers exist."""
    rng = np.random.default_rng(7)
    pool = np.array([np.nan, np.inf, -np.inf, 0.0, -0.0, 1.0, -1.0, 2.5], dtype=np.float32)
    for _ in range(400):
        E = int(rng.integers(3, 9))
        k = int(rng.integers(1, E + 1))
        l = rng.choice(pool, size=(1, E)).astype(np.float32)
        def key(e):
            v = l[0, e]
            return (bool(np.isnan(v)), 0.0 if np.isnan(v) else -float(v), e)
        order = sorted(range(E), key=key)
        with np.errstate(invalid="ignore", over="ignore"):  # the weights of such rows are not checked here
            ids, _ = moe.topk_softmax(l, k)
        assert list(ids[0]) == order[:k], (l, k)


def test_swiglu_clamp_against_torch_silu():
    g = np.array([-50, -3, 0, 2.5, 9.99, 10, 11, 1e4])
    u = np.array([-1e3, -10, -9.5, 0, 3, 10, 10.5, 50])
    L = 10.0
    got = moe.swiglu(g, u, L)
    ref = (F.silu(torch.tensor(g).clamp(max=L)) * torch.tensor(u).clamp(-L, L)).numpy()
    assert np.allclose(got, ref, rtol=1e-15, atol=1e-300)
    assert got[-1] == pytest.approx(10.0 / (1 + np.exp(-10.0)) * 10.0)


def _tiny_setup(seed=sg.EVAL_SEED):
    wl = sg.TINY
    x = sg.activations_bf16(wl, seed)
    wr = sg.router_bf16(wl)
    experts = [moe.quantize_expert(sg.expert_w1_f32(wl, e), sg.expert_w2_f32(wl, e)) for e in range(wl.E)]
    return wl, x, wr, experts


def test_identity_codec_layer_is_the_textbook_dense_moe():
    wl, x, wr, experts = _tiny_setup()
    l = moe.router_logits(x, wr)
    ids, w = moe.topk_softmax(l, wl.k)
    y = moe.moe_tokens(x, ids, w, lambda e: experts[e], 1.0, 1.0, wl.swiglu_limit, quantize_activations=False)
    # textbook: every expert on every token, then gather the top-k and weight
    xt = torch.from_numpy(moe.bf16_to_f64(x))
    W1 = torch.stack([torch.from_numpy(nvfp4.dequantize(q.w1_q, q.w1_sf, q.w1_gs)) for q in experts])
    W2 = torch.stack([torch.from_numpy(nvfp4.dequantize(q.w2_q, q.w2_sf, q.w2_gs)) for q in experts])
    gu = torch.einsum("th,eoh->teo", xt, W1)
    I = wl.I
    h = F.silu(gu[..., :I].clamp(max=wl.swiglu_limit)) * gu[..., I:].clamp(-wl.swiglu_limit, wl.swiglu_limit)
    o = torch.einsum("tei,ehi->teh", h, W2).float().bfloat16().double()   # l2_out is BF16 ("Data Flow")
    lt = torch.from_numpy(l.astype(np.float64))
    tv, ti = torch.topk(lt, wl.k, dim=1)
    wt = torch.softmax(tv, dim=1)
    ref = (wt[..., None] * torch.gather(o, 1, ti[..., None].expand(-1, -1, wl.H))).sum(1)
    ref_bits = sg.f32_to_bf16_bits(ref.numpy().astype(np.float32))
    assert (y == ref_bits).mean() > 0.999
    assert np.allclose(sg.bf16_bits_to_f32(y), sg.bf16_bits_to_f32(ref_bits), rtol=1e-2, atol=1e-6)


def _naive_layer(x_bits, ids, w, experts, gs1, gs2, L):
    """Second path: dense fp64 matrices from an element-by-element decode, plain loops."""
    from oracle import codecs
    H = x_bits.shape[1]
    out = []
    for t in range(x_bits.shape[0]):
        xf = sg.bf16_bits_to_f32(x_bits[t:t + 1])
        q, sf = nvfp4.quantize_rows(xf, gs1)
        xt = [float(codecs.e2m1_decode(q[0, i])) * float(codecs.e4m3_decode(sf[0, i // 16])) / float(gs1) for i in range(H)]
        acc = [0.0] * H
        for j in range(ids.shape[1]):
            qe = experts[int(ids[t, j])]
            I = qe.w2_q.shape[1]
            def w1(r, c):
                return float(codecs.e2m1_decode(qe.w1_q[r, c])) * float(codecs.e4m3_decode(qe.w1_sf[r, c // 16])) / float(qe.w1_gs)
            def w2(r, c):
                return float(codecs.e2m1_decode(qe.w2_q[r, c])) * float(codecs.e4m3_decode(qe.w2_sf[r, c // 16])) / float(qe.w2_gs)
            gate = [sum(w1(i, c) * xt[c] for c in range(H)) for i in range(I)]
            up = [sum(w1(I + i, c) * xt[c] for c in range(H)) for i in range(I)]
            h = moe.swiglu(np.array(gate), np.array(up), L).astype(np.float32).reshape(1, I)
            q2, s2 = nvfp4.quantize_rows(h, gs2)
            ht = [float(codecs.e2m1_decode(q2[0, c])) * float(codecs.e4m3_decode(s2[0, c // 16])) / float(gs2) for c in range(I)]
            for r in range(H):   # each pair row leaves the second GEMM in BF16 ("Data Flow": l2_out)
                o_r = sum(w2(r, c) * ht[c] for c in range(I))
                acc[r] += w[t, j] * float(torch.tensor(o_r, dtype=torch.float64).float().bfloat16().double())
        out.append(acc)
    return np.array(out)


@pytest.mark.slow
def test_tiny_layer_against_naive_second_path():
    wl, x, wr, experts = _tiny_setup()
    l = moe.router_logits(x, wr)
    ids, w = moe.topk_softmax(l, wl.k)
    gs1, gs2 = moe.calibrate(sg.activations_bf16(wl, sg.WARMUP_SEED),
                             moe.topk_softmax(moe.router_logits(sg.activations_bf16(wl, sg.WARMUP_SEED), wr), wl.k)[0],
                             lambda e: experts[e], wl.swiglu_limit)
    rows = [0, 5, 15]
    y = moe.moe_tokens(x[rows], ids[rows], w[rows], lambda e: experts[e], gs1, gs2, wl.swiglu_limit)
    ref = _naive_layer(x[rows], ids[rows], w[rows], experts, gs1, gs2, wl.swiglu_limit)
    got = sg.bf16_bits_to_f32(y).astype(np.float64)
    assert np.allclose(got, ref, rtol=2**-8, atol=1e-9)
    assert (y == sg.f32_to_bf16_bits(ref.astype(np.float32))).mean() > 0.99


def test_calibration_scales_come_from_the_warmup_batch():
    wl, _, wr, experts = _tiny_setup()
    xw = sg.activations_bf16(wl, sg.WARMUP_SEED)
    ids, _ = moe.topk_softmax(moe.router_logits(xw, wr), wl.k)
    gs1, gs2 = moe.calibrate(xw, ids, lambda e: experts[e], wl.swiglu_limit)
    assert gs1 == nvfp4.global_scale(np.abs(sg.bf16_bits_to_f32(xw)).max())
    # with gs2 the warmup h has no saturated block scale and reaches the top code somewhere
    xt = nvfp4.dequantize(*nvfp4.quantize_rows(sg.bf16_bits_to_f32(xw), gs1), gs1)
    hs = [moe.expert_hidden(experts[e], xt[np.nonzero(ids == e)[0]], wl.swiglu_limit) for e in np.unique(ids)]
    h = np.concatenate(hs).astype(np.float32)
    assert float(np.abs(h).max()) * float(gs2) == pytest.approx(2688.0, rel=1e-6)


def test_expert_parallel_parts_sum_to_the_layer():
    """The rank parts of an EP split (masked pairs left out) sum to the whole layer, before the final bf16
    rounding (each pair row already in BF16, as the second GEMM returns it)."""
    wl = sg.TINY
    x = sg.activations_bf16(wl, sg.EVAL_SEED, T=6)
    ids, w = moe.topk_softmax(moe.router_logits(x, sg.router_bf16(wl), None), wl.k)
    cache = {}

    def expert(e):
        if e not in cache:
            cache[e] = moe.quantize_expert(sg.expert_w1_f32(wl, e), sg.expert_w2_f32(wl, e))
        return cache[e]
    gs1, gs2 = np.float32(200.0), np.float32(300.0)
    xf = sg.bf16_bits_to_f32(x).astype(np.float64)

    def layer_sum(ids_local, first):
        """sum_j w_j o_j over held pairs, in fp64 (the layer before its final bf16 rounding)."""
        q, s = nvfp4.quantize_rows(xf.astype(np.float32), gs1)
        xt = nvfp4.dequantize(q, s, gs1)
        acc = np.zeros((x.shape[0], wl.H))
        for t in range(x.shape[0]):
            for j in range(wl.k):
                if ids_local[t, j] < 0:
                    continue
                qe = expert(first + int(ids_local[t, j]))
                h = moe.expert_hidden(qe, xt[t:t + 1], wl.swiglu_limit)
                acc[t] += w[t, j] * moe.l2_out_bf16(moe.expert_out(qe, h, gs2))[0]
        return acc

    full = layer_sum(ids, 0)
    parts = sum(layer_sum(layout.local_ids(ids, f, 4), f) for f in (0, 4))
    assert np.allclose(parts, full, rtol=1e-12, atol=1e-15)
    # and moe_tokens with a masked routing rounds that part
    part0 = moe.moe_tokens(x, layout.local_ids(ids, 0, 4), w, lambda l: expert(l), gs1, gs2, wl.swiglu_limit)
    ref0 = moe.f32_to_bf16_bits(layer_sum(layout.local_ids(ids, 0, 4), 0).astype(np.float32))
    assert (part0 == ref0).all()
