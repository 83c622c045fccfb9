"""GPU: the weight prep (fp4moe_quantize_weights) against the oracle's quantiser.

Codes, swizzled scales and per-expert global scales are compared bit for
bit, after undoing the documented pre-tiling and the W1 gate/up row order.
"""
import numpy as np
import pytest

import synthgen as sg
from helpers import OracleExperts, ensure_built, make_layer, untile_weights
from oracle import nvfp4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _w1_kernel_rows(I):
    """kernel row -> logical W13 row (gate rows [0, I), up rows [I, 2I))."""
    o = np.arange(2 * I)
    f = 64 * (o // 128) + o % 64
    return np.where((o % 128) < 64, f, I + f)


def check_experts(wl, layer, experts_to_check):
    H, I, E = wl.H, wl.I, wl.E
    W = layer.weights
    w1c = untile_weights(W.w1_fp4.cpu().numpy(), E * 2 * I, H // 2, 2 * I).reshape(E, 2 * I, H // 2)
    w1s = W.w1_sf.cpu().numpy().reshape(E, -1)
    w2c = untile_weights(W.w2_fp4.cpu().numpy(), E * H, I // 2, H).reshape(E, H, I // 2)
    w2s = W.w2_sf.cpu().numpy().reshape(E, -1)
    gw1 = W.gw1.cpu().numpy()
    gw2 = W.gw2.cpu().numpy()
    oracle = OracleExperts(wl)
    rows = _w1_kernel_rows(I)
    for e in experts_to_check:
        q = oracle(e)
        assert gw1[e] == q.w1_gs and gw2[e] == q.w2_gs
        assert (w1c[e] == nvfp4.pack_codes(q.w1_q)[rows]).all()
        assert (nvfp4.unswizzle(w1s[e], 2 * I, H // 16) == q.w1_sf[rows]).all()
        assert (w2c[e] == nvfp4.pack_codes(q.w2_q)).all()
        assert (nvfp4.unswizzle(w2s[e], H, I // 16) == q.w2_sf).all()


def test_weight_prep_tiny_all_experts():
    wl = sg.TINY
    check_experts(wl, make_layer(wl, 16), range(wl.E))


def test_weight_prep_dsv4_sampled_experts():
    wl = sg.DSV4_DECODE
    check_experts(wl, make_layer(wl, 64), [0, 77, 255])
