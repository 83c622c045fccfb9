"""GPU: stale activation scales are detected on the device, and gs2 is refreshed there.

"Current Bug: CuTeDSLMoERunner", "Bug 5" and "Bug 6": activation global
scales fixed in a warm-up pass go stale when later activations outgrow them,
and the E4M3 block scales then saturate at 448 (an L2 amax of about 286
against a scale taken from a much smaller range). Here, on the tiny workload:

* the warm-up batch itself raises no saturation flag, and refreshing gs2 from
  its own running amax|h| gives back the calibrated gs2 bit for bit;
* a batch 16 times the warm-up's (with its own gs1 from fp4moe_batch_gs1)
  raises FP4MOE_SAT_L2 and not FP4MOE_SAT_L1; the oracle confirms that some of
  its h blocks saturate under the stale gs2 and that the running amax is the
  batch's amax|h|;
* fp4moe_refresh_gs2 then gives the oracle's gs2 for that amax, and the
  alpha2 table RN(1 / RN(gs2 * gw2)); the rerun raises no flag and matches
  the oracle's layer under the new scales within the float bar;
* fp4moe_calibrate captured in a CUDA graph gives the eager scales, bit for bit.
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


def _forward(layer, x_bits):
    import torch
    y = torch.empty(x_bits.shape[0], layer.cfg.hidden, dtype=torch.bfloat16, device="cuda")
    layer.forward(bits_to_torch(x_bits), y)
    torch.cuda.synchronize()
    assert layer.read_error() == 0
    return torch_to_bits(y)


def test_stale_gs2_is_flagged_and_refreshed():
    from block_scaled_fp4_top_gb300 import _lib
    wl = sg.TINY
    layer = make_layer(wl, wl.T)
    experts = OracleExperts(wl)
    wr = sg.router_bf16(wl)
    xw = sg.activations_bf16(wl, sg.WARMUP_SEED)
    layer.calibrate(bits_to_torch(xw))
    gs2_cal = layer.gs2.clone()
    assert layer.read_scale_status() == (0, 0.0)          # calibration leaves the hot-path words alone
    # the warm-up batch: inside the scales it set
    _forward(layer, xw)
    flags, amax_w = layer.read_scale_status()
    assert flags == 0 and amax_w > 0
    layer.refresh_gs2()                                      # the same h as the calibration: the same gs2
    assert float(layer.gs2.item()) == float(gs2_cal.item())
    assert layer.read_scale_status()[1] == 0.0               # the refresh clears the running amax

    # a batch 16x the warm-up's: exact in bf16 (an exponent shift)
    x16f = sg.bf16_bits_to_f32(xw) * np.float32(16.0)
    x16 = sg.f32_to_bf16_bits(x16f)
    assert np.array_equal(sg.bf16_bits_to_f32(x16), x16f)
    layer.batch_gs1(bits_to_torch(x16))
    gs1_16 = moe.activation_scale(x16)
    assert float(layer.gs1.item()) == float(gs1_16)
    y_stale = _forward(layer, x16)
    flags, amax_gpu = layer.read_scale_status()
    assert flags == _lib.SAT_L2, flags
    # the oracle: this batch's h, its amax, and blocks that saturate under the stale gs2
    ids, w = moe.topk_softmax(moe.router_logits(x16, wr), wl.k)
    xt = moe.dequantized_activations(x16, gs1_16)
    hs = [moe.expert_hidden(experts(e), xt[tt], wl.swiglu_limit) for e, (tt, _) in moe.routed_rows(ids).items()]
    amax16 = max(moe.hidden_amax(experts(e), xt[tt], wl.swiglu_limit) for e, (tt, _) in moe.routed_rows(ids).items())
    assert amax_gpu == pytest.approx(amax16, rel=1e-5)
    stale = np.float32(gs2_cal.item())
    assert any((nvfp4.block_scales(h.astype(np.float32), stale) > nvfp4.E4M3_SATURATES_ABOVE).any() for h in hs)
    # refresh: gs2 from the running amax, alpha2 from it, then the batch fits
    layer.refresh_gs2()
    gs2_new = np.float32(layer.gs2.item())
    assert gs2_new == pytest.approx(float(nvfp4.global_scale(np.float32(amax16))), rel=1e-5)
    gw2 = layer.weights.gw2.cpu().numpy()
    alpha2 = (np.float32(1.0) / (gs2_new * gw2).astype(np.float32)).astype(np.float32)
    assert np.array_equal(layer.alpha2.cpu().numpy(), alpha2)
    y_new = _forward(layer, x16)
    assert layer.read_scale_status()[0] == 0
    ref = moe.moe_tokens(x16, ids, w, experts, gs1_16, nvfp4.global_scale(np.float32(amax16)), wl.swiglu_limit)
    float_parity(sg.bf16_bits_to_f32(y_new), sg.bf16_bits_to_f32(ref), bf16=True)
    # the stale run really lost range: it is further from that reference than the refreshed one
    err = lambda y: np.linalg.norm(sg.bf16_bits_to_f32(y) - sg.bf16_bits_to_f32(ref))
    assert err(y_stale) > err(y_new)


def test_refresh_with_no_h_leaves_the_scales():
    wl = sg.TINY
    layer = make_layer(wl, wl.T)
    layer.set_global_scales(3.0, 5.0)
    a2 = layer.alpha2.clone()
    layer.refresh_gs2()
    assert float(layer.gs2.item()) == 5.0 and bool((layer.alpha2 == a2).all())


def test_calibrate_captured_in_a_graph_matches_eager():
    import torch
    from block_scaled_fp4_top_gb300 import api
    wl = sg.DSV4_DECODE
    layer = make_layer(wl, wl.T)
    xw = bits_to_torch(sg.activations_bf16(wl, sg.WARMUP_SEED))
    layer.calibrate(xw)                                      # eager, and every first-call set-up
    torch.cuda.synchronize()
    gs1_g = torch.zeros(1, dtype=torch.float32, device="cuda")
    gs2_g = torch.zeros(1, dtype=torch.float32, device="cuda")
    W = layer.weights
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            api.fp4moe_calibrate(layer.cfg, wl.T, xw, layer.router_w, layer.router_bias, W.w1_fp4, W.w1_sf, W.gw1,
                                 gs1_g, gs2_g, layer.ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        gs1_g.zero_()
        gs2_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert float(gs1_g.item()) == float(layer.gs1.item())
        assert float(gs2_g.item()) == float(layer.gs2.item())
    assert layer.read_error() == 0
