"""GPU: the whole layer (moe_forward) and its calibration against the oracle.

* tiny workload: every token, T in {16, 1, 5, 13};
* DeepSeek-V4-Flash decode (T = 64): every token, with the oracle's own
  warm-up scales (gs1 bit-equal to the library's, gs2 within 1e-5);
* Zipf prefill (T = 8192): top-k ids of every token, and the output rows of
  320 tokens: 256 seeded ones plus tokens routed to the three most popular
  experts (over 1000 tokens each) and to experts whose rows fill a single
  partial 128-row tile.
Also: the empty batch, CUDA-graph capture with changed-input replay, and
determinism. The oracle's per-expert work runs on the test-side worker pool
(tests/oracle_pool.py); every value it returns is the oracle's.
"""
import numpy as np
import pytest

import synthgen as sg
from helpers import (OracleExperts, assert_sched_counters_zero, bits_to_torch, ensure_built, float_parity,
                     make_layer, torch_to_bits)
from oracle import moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _calibrated(wl, max_tokens, warm_T=None):
    layer = make_layer(wl, max_tokens)
    xw = sg.activations_bf16(wl, sg.WARMUP_SEED, T=warm_T or wl.T)
    layer.calibrate(bits_to_torch(xw))
    return layer, xw


def _oracle_scales(wl, xw, experts):
    ids, _ = moe.topk_softmax(moe.router_logits(xw, sg.router_bf16(wl), sg.router_bias_f32(wl)), wl.k)
    return moe.calibrate(xw, ids, experts, wl.swiglu_limit)


def _oracle_rows(wl, x_bits, rows, experts, gs1, gs2):
    l = moe.router_logits(x_bits[rows], sg.router_bf16(wl), sg.router_bias_f32(wl))
    ids, w = moe.topk_softmax(l, wl.k)
    y = moe.moe_tokens(x_bits[rows], ids, w, experts, gs1, gs2, wl.swiglu_limit)
    return sg.bf16_bits_to_f32(y), ids


def _forward(layer, wl, x_bits):
    import torch
    T = x_bits.shape[0]
    y = torch.empty(max(T, 1), wl.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(max(T, 1) * wl.k, dtype=torch.int32, device="cuda")
    x = bits_to_torch(x_bits) if T else torch.zeros(1, wl.H, dtype=torch.bfloat16, device="cuda")
    layer.forward(x[:T] if T else x, y, ids, None)
    torch.cuda.synchronize()
    assert layer.read_error() == 0
    assert_sched_counters_zero(layer.ws)
    return sg.bf16_bits_to_f32(torch_to_bits(y))[:T], ids.cpu().numpy()[: T * wl.k].reshape(T, wl.k)


@pytest.fixture(scope="module")
def tiny():
    wl = sg.TINY
    layer, xw = _calibrated(wl, wl.T)
    experts = OracleExperts(wl)
    gs1, gs2 = _oracle_scales(wl, xw, experts)
    return wl, layer, experts, gs1, gs2


def test_tiny_calibration(tiny):
    wl, layer, experts, gs1, gs2 = tiny
    assert float(layer.gs1.item()) == float(gs1)  # amax is exact: bit-equal
    assert float(layer.gs2.item()) == pytest.approx(float(gs2), rel=1e-5)


@pytest.mark.parametrize("T", [16, 1, 5, 13])
def test_tiny_forward_all_tokens(tiny, T):
    wl, layer, experts, gs1, gs2 = tiny
    x = sg.activations_bf16(wl, sg.EVAL_SEED, T=T)
    y, ids = _forward(layer, wl, x)
    # the oracle runs with the GPU's calibrated scales' values taken from its own warmup
    ref, ids_ref = _oracle_rows(wl, x, np.arange(T), experts, gs1, gs2)
    assert (ids == ids_ref).all()
    float_parity(y, ref, bf16=True)


def test_nan_token_sets_the_nan_bit_and_spares_the_others(tiny):
    """A NaN in one token's x: the oracle has no codes for it (its encoder rejects NaN), so the library raises
    FP4MOE_ERR_NAN from the quantiser, beside FP4MOE_ERR_EXPERT_ID from the router (a NaN logit ranks nowhere,
    so the token gets ids 0 and weights 0). Rows of an MMA are independent, so every other token's output
    equals, bit for bit, that of the same batch with the NaN token's row zeroed."""
    import torch
    from block_scaled_fp4_top_gb300 import _lib
    wl, layer, _, _, _ = tiny
    x = sg.activations_bf16(wl, sg.EVAL_SEED, T=wl.T)
    x_zero, x_nan = x.copy(), x.copy()
    x_zero[3] = 0
    x_nan[3, 17] = 0x7FC0                                   # bf16 quiet NaN
    with pytest.raises(ValueError):
        moe.dequantized_activations(x_nan[3:4], np.float32(1.0))
    y0, _ = _forward(layer, wl, x_zero)
    y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device="cuda")
    layer.forward(bits_to_torch(x_nan), y)
    torch.cuda.synchronize()
    assert layer.read_error() == _lib.ERR_NAN | _lib.ERR_EXPERT_ID
    y1 = sg.bf16_bits_to_f32(torch_to_bits(y))
    others = np.arange(wl.T) != 3
    assert np.array_equal(y1[others].view(np.uint32), y0[others].view(np.uint32))


def test_empty_batch(tiny):
    wl, layer, _, _, _ = tiny
    y, _ = _forward(layer, wl, np.zeros((0, wl.H), np.uint16))
    assert y.shape == (0, wl.H)


@pytest.fixture(scope="module")
def dsv4():
    wl = sg.DSV4_DECODE
    layer, xw = _calibrated(wl, 4096)
    experts = OracleExperts(wl)
    return wl, layer, experts, xw


def test_dsv4_decode_all_tokens(dsv4, oracle_svc):
    wl, layer, experts, xw = dsv4
    gs1, gs2 = oracle_svc.calibrate(wl, xw)
    assert float(layer.gs1.item()) == float(gs1)  # the amax is exact: bit-equal
    assert float(layer.gs2.item()) == pytest.approx(float(gs2), rel=1e-5)
    x = sg.activations_bf16(wl, sg.EVAL_SEED, T=wl.T)
    y, ids = _forward(layer, wl, x)
    (y_ref, ids_ref, _), = oracle_svc.layer(wl, [x], gs1, gs2)
    assert (ids == ids_ref).all()
    float_parity(y, sg.bf16_bits_to_f32(y_ref), bf16=True)


def test_dsv4_determinism_and_graph_replay(dsv4):
    import torch
    wl, layer, _, _ = dsv4
    from block_scaled_fp4_top_gb300 import api
    for T in (1, 8, 64):
        x_static = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")
        y_static = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")
        x_static.copy_(bits_to_torch(sg.activations_bf16(wl, sg.REPLAY_SEED0, T=T)))
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            layer.forward(x_static, y_static)          # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer.forward(x_static, y_static)
        for i in range(3):
            xb = sg.activations_bf16(wl, sg.REPLAY_SEED0 + i, T=T)
            x_static.copy_(bits_to_torch(xb))
            g.replay()
            torch.cuda.synchronize()
            got = torch_to_bits(y_static)
            y_eager, _ = _forward(layer, wl, xb)
            assert (got == sg.f32_to_bf16_bits(y_eager)).all(), f"replay {i} at T={T} differs from eager"
        assert layer.read_error() == 0


def _prefill_rows(ids_ref, E, rng):
    """256 seeded tokens, 8 tokens of each of the three most popular experts, and one token of each expert
    (up to 32) whose rows fill a single partial 128-row tile."""
    counts = np.bincount(ids_ref.reshape(-1), minlength=E)
    rows = set(rng.choice(ids_ref.shape[0], 256, replace=False).tolist())
    for e in np.argsort(-counts, kind="stable")[:3]:
        tok = np.nonzero((ids_ref == e).any(axis=1))[0]
        rows.update(rng.choice(tok, 8, replace=False).tolist())
    partial = [e for e in range(E) if 0 < counts[e] < 128][:32]
    for e in partial:
        rows.add(int(np.nonzero((ids_ref == e).any(axis=1))[0][0]))
    return np.array(sorted(rows)), counts, partial


def test_zipf_prefill_many_tokens(oracle_svc):
    wl = sg.DSV4_PREFILL_ZIPF
    layer, xw = _calibrated(wl, wl.T)
    gs1, gs2 = oracle_svc.calibrate(wl, xw)
    assert float(layer.gs1.item()) == float(gs1)
    assert float(layer.gs2.item()) == pytest.approx(float(gs2), rel=1e-5)
    x = sg.activations_bf16(wl, sg.EVAL_SEED, T=wl.T)
    y, ids = _forward(layer, wl, x)
    assert np.isfinite(y).all()
    ids_ref, _ = moe.topk_softmax(moe.router_logits(x, sg.router_bf16(wl), sg.router_bias_f32(wl)), wl.k)
    assert (ids == ids_ref).all()                        # every token's routing, bit-exact
    rows, counts, partial = _prefill_rows(ids_ref, wl.E, np.random.default_rng(17))
    assert counts.max() > 1000 and (counts == 0).sum() >= 16 and len(partial) > 0
    assert len(rows) >= 256
    (y_ref, ids_rows, _), = oracle_svc.layer(wl, [x[rows]], gs1, gs2)
    assert (ids_rows == ids_ref[rows]).all()
    float_parity(y[rows], sg.bf16_bits_to_f32(y_ref), bf16=True)
    # Every token's row depends on that token alone, and each accumulation runs in a fixed K order. So the
    # leading tokens of the batch come out bit for bit the same under every schedule and tile shape:
    # T = 8192 (dynamic chunks, 128 x 256 tiles), 512 (static with its tail pool, 128 x 256), 64 (static with
    # its tail pool, 128 x 128) and 1 (static, no pool).
    for T in (512, 64, 1):
        y_T, ids_T = _forward(layer, wl, x[:T])
        assert (ids_T == ids[:T]).all()
        assert np.array_equal(y_T, y[:T]), f"T={T}: rows differ from the same tokens inside the T=8192 batch"
