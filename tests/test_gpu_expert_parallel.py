"""GPU: expert parallelism on one GPU ("Current Bug", "Bug 8", "Bug 13", "EP Configuration").

The layer holds experts [ep_first, ep_first + ep_count) of the router's 256.
The router still scores all of them and reports global ids. The layout maps
them to local ids and masks the pairs held elsewhere (slot -1). The output is
this rank's part of the layer.

Checks:
* DeepSeek-V4-Flash decode with 48 local experts starting at 96, the pages'
  "in practice 48": global ids bit-exact; local counts, offsets, padded
  offsets, slots and rows bit-exact against the oracle's remap; output rows
  within the float bar against the oracle's masked layer; and warm-up
  calibration over local ids only, so gs2 is not the 0 of "Bug 13".
* The tiny shape split over two ranks: each rank's part against the oracle,
  and the two parts summed against the whole layer.
"""
import numpy as np
import pytest
import torch

import synthgen as sg
from helpers import OracleExperts, bits_to_torch, ensure_built, float_parity, torch_to_bits
from oracle import layout, moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def ep_layer(wl, first, count, max_tokens):
    from block_scaled_fp4_top_gb300 import api
    from synthgen import gpu as sgpu
    cfg = api.config(wl.H, wl.I, wl.E, wl.k, max_tokens, wl.swiglu_limit, ep_first=first, ep_count=count)
    layer = api.MoELayer(cfg)
    for e0 in range(0, count, 16):
        n = min(16, count - e0)
        layer.quantize_weights(1, e0, sgpu.expert_w1(wl, first + e0, n))
        layer.quantize_weights(2, e0, sgpu.expert_w2(wl, first + e0, n))
    layer.set_router(sgpu.router(wl), None)
    torch.cuda.synchronize()
    return cfg, layer


def forward(layer, wl, x_bits):
    T = x_bits.shape[0]
    y = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(T * wl.k, dtype=torch.int32, device="cuda")
    layer.forward(bits_to_torch(x_bits), y, ids)
    torch.cuda.synchronize()
    assert layer.read_error() == 0
    return sg.bf16_bits_to_f32(torch_to_bits(y)).astype(np.float64), ids.cpu().numpy().reshape(T, wl.k)


def test_dsv4_decode_48_local_experts():
    from block_scaled_fp4_top_gb300 import api
    wl = sg.DSV4_DECODE
    first, count = 96, 48
    cfg, layer = ep_layer(wl, first, count, wl.T)
    xw = sg.activations_bf16(wl, sg.WARMUP_SEED)
    layer.calibrate(bits_to_torch(xw))
    experts = OracleExperts(wl)
    wr = sg.router_bf16(wl)
    ids_w, _ = moe.topk_softmax(moe.router_logits(xw, wr, None), wl.k)
    gs1_ref, gs2_ref = moe.calibrate(xw, layout.local_ids(ids_w, first, count), lambda l: experts(first + l),
                                     wl.swiglu_limit)
    gs1, gs2 = np.float32(layer.gs1.item()), np.float32(layer.gs2.item())
    assert gs1 == gs1_ref and gs2 > 0 and gs2 == pytest.approx(float(gs2_ref), rel=1e-5)

    x = sg.activations_bf16(wl, sg.EVAL_SEED)
    # the routing outputs of the EP layer, through moe_route
    cap = api.capacity_rows(cfg, wl.T)
    i32 = dict(dtype=torch.int32, device="cuda")
    o = dict(logits=torch.empty(wl.T, wl.E, device="cuda"), ids=torch.empty(wl.T * wl.k, **i32),
             w=torch.empty(wl.T * wl.k, device="cuda"), counts=torch.empty(count, **i32),
             offsets=torch.empty(count, **i32), poff=torch.empty(count, **i32), slot=torch.empty(wl.T * wl.k, **i32),
             por=torch.full((cap,), -7, **i32))
    api.moe_route(cfg, wl.T, bits_to_torch(x), layer.router_w, None, o["logits"], o["ids"], o["w"], o["counts"],
                  o["offsets"], o["poff"], o["slot"], o["por"], layer.ws)
    torch.cuda.synchronize()
    ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x, wr, None), wl.k)
    assert (o["ids"].cpu().numpy().reshape(wl.T, wl.k) == ids_ref).all()   # global ids
    loc = layout.local_ids(ids_ref, first, count)
    L = layout.slots(loc, count)
    assert (o["counts"].cpu().numpy() == L["counts"]).all()
    assert (o["offsets"].cpu().numpy() == L["offsets"]).all()
    assert (o["poff"].cpu().numpy() == L["padded_offsets"]).all()
    assert (o["slot"].cpu().numpy() == L["slot_of_pair"]).all()
    assert (o["por"].cpu().numpy()[:L["R"]] == L["pair_of_row"]).all()
    assert api.capacity_rows(cfg, wl.T) == layout.capacity_rows(wl.T, wl.k, count)

    y, ids = forward(layer, wl, x)
    assert (ids == ids_ref).all()
    rows = np.array([0, 21, 42, 63])
    y_ref = moe.moe_tokens(x[rows], loc[rows], w_ref[rows], lambda l: experts(first + l), gs1, gs2, wl.swiglu_limit)
    float_parity(y[rows], sg.bf16_bits_to_f32(y_ref), bf16=True)


def test_tiny_two_rank_split_sums_to_the_layer():
    wl = sg.TINY
    x = sg.activations_bf16(wl, sg.EVAL_SEED)
    xw = sg.activations_bf16(wl, sg.WARMUP_SEED)
    experts = OracleExperts(wl)
    ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x, sg.router_bf16(wl), None), wl.k)
    # one pair of activation scales for every rank: those of the whole layer's warm-up batch
    ids_w, _ = moe.topk_softmax(moe.router_logits(xw, sg.router_bf16(wl), None), wl.k)
    gs1, gs2 = moe.calibrate(xw, ids_w, experts, wl.swiglu_limit)
    total = np.zeros((wl.T, wl.H))
    parts = []
    for first in (0, 4):
        _, layer = ep_layer(wl, first, 4, wl.T)
        layer.set_global_scales(float(gs1), float(gs2))
        y, ids = forward(layer, wl, x)
        assert (ids == ids_ref).all()
        loc = layout.local_ids(ids_ref, first, 4)
        y_ref = moe.moe_tokens(x, loc, w_ref, lambda l: experts(first + l), gs1, gs2, wl.swiglu_limit)
        float_parity(y, sg.bf16_bits_to_f32(y_ref), bf16=True)
        total += y
        parts.append(y)
    y_full = moe.moe_tokens(x, ids_ref, w_ref, experts, gs1, gs2, wl.swiglu_limit)
    float_parity(total, sg.bf16_bits_to_f32(y_full), bf16_terms=parts)
