"""GPU: the L1 activation global scale taken from the batch in hand (fp4moe_batch_gs1).

A warm-up calibration fixes gs1 = RN(2688 / amax) of the warm-up batch
("Current Bug", "Bug 5" and "Bug 6"). A batch sixteen times larger then
saturates its E4M3 block scales at 448: the calibration-drift failure mode.
fp4moe_batch_gs1 recomputes gs1 and the alpha1 table from the batch, on the
device, in one launch, with no host synchronisation. Checks:
* gs1 and alpha1 equal, bit for bit, the oracle's global scale of the batch and
  RN(1 / RN(gs1 * gw1[e]));
* the layer then meets the float bar against the oracle using that scale;
* the stale warm-up scale misses the same oracle by far more.
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


def _forward(layer, x, wl):
    import torch
    y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device="cuda")
    layer.forward(x, y)
    torch.cuda.synchronize()
    assert layer.read_error() == 0
    return sg.bf16_bits_to_f32(torch_to_bits(y)).astype(np.float64)


def test_batch_gs1_matches_the_oracle_and_removes_saturation():
    import torch
    wl = sg.TINY
    layer = make_layer(wl, wl.T)
    layer.calibrate(bits_to_torch(sg.activations_bf16(wl, sg.WARMUP_SEED)))
    gs1_warm = np.float32(layer.gs1.item())
    # 16x the evaluation batch: a power of two, so exact in bf16
    xf = sg.bf16_bits_to_f32(sg.activations_bf16(wl, sg.EVAL_SEED)) * np.float32(16.0)
    x_bits = sg.f32_to_bf16_bits(xf)
    x = bits_to_torch(x_bits)
    y_stale = _forward(layer, x, wl)

    layer.batch_gs1(x)
    torch.cuda.synchronize()
    gs1 = np.float32(layer.gs1.item())
    assert gs1 == nvfp4.global_scale(np.abs(xf).max()) and gs1 < gs1_warm
    gw1 = layer.weights.gw1.cpu().numpy()
    alpha_ref = (np.float32(1.0) / (gs1 * gw1).astype(np.float32)).astype(np.float32)
    assert np.array_equal(layer.alpha1.cpu().numpy().view(np.uint32), alpha_ref.view(np.uint32))
    assert layer.read_error() == 0
    y_dyn = _forward(layer, x, wl)

    ids, w = moe.topk_softmax(moe.router_logits(x_bits, sg.router_bf16(wl), None), wl.k)
    gs2 = np.float32(layer.gs2.item())
    y_ref = sg.bf16_bits_to_f32(moe.moe_tokens(x_bits, ids, w, OracleExperts(wl), gs1, gs2, wl.swiglu_limit))
    rel_dyn, _ = float_parity(y_dyn, y_ref, bf16=True)
    rel_stale = np.linalg.norm(y_stale - y_ref) / np.linalg.norm(y_ref)
    assert rel_stale > 4 * max(rel_dyn, 1e-3), (rel_stale, rel_dyn)
