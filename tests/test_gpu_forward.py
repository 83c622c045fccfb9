"""GPU: the whole layer (moe_forward) and its calibration against the oracle,
at the tiny workload (all tokens) and the DeepSeek-V4-Flash decode and Zipf
prefill workloads (sampled tokens). Also: ragged and empty T, CUDA-graph
capture with changed-input replay, and determinism.
"""
import numpy as np
import pytest

import synthgen as sg
from helpers import OracleExperts, bits_to_torch, ensure_built, float_parity, make_layer, torch_to_bits
from oracle import moe, nvfp4

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
    float_parity(y, ref)


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


def test_dsv4_decode_sampled_tokens(dsv4):
    wl, layer, experts, xw = dsv4
    x = sg.activations_bf16(wl, sg.EVAL_SEED, T=wl.T)
    y, ids = _forward(layer, wl, x)
    assert np.isfinite(y).all()
    gs1 = float(layer.gs1.item())
    xf = sg.bf16_bits_to_f32(xw)
    assert gs1 == float(nvfp4.global_scale(np.abs(xf).max()))
    gs2 = np.float32(layer.gs2.item())  # gs2 check vs the oracle's own warmup is in the tiny test
    rows = np.array([0, 21, 42, 63])
    ref, ids_ref = _oracle_rows(wl, x, rows, experts, np.float32(gs1), gs2)
    assert (ids[rows] == ids_ref).all()
    float_parity(y[rows], ref)


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


def test_zipf_prefill_sampled_tokens():
    wl = sg.DSV4_PREFILL_ZIPF
    layer, xw = _calibrated(wl, wl.T)
    experts = OracleExperts(wl)
    x = sg.activations_bf16(wl, sg.EVAL_SEED, T=wl.T)
    y, ids = _forward(layer, wl, x)
    assert np.isfinite(y).all()
    rows = np.array([0, 4095, 8191])
    ref, ids_ref = _oracle_rows(wl, x, rows, experts, np.float32(layer.gs1.item()), np.float32(layer.gs2.item()))
    assert (ids[rows] == ids_ref).all()
    float_parity(y[rows], ref)
