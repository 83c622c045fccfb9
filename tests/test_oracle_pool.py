"""The test-side oracle pool gives the serial oracle's results bit for bit (tiny NVFP4 and MXFP4 layers), so
the full-size GPU parity tests that use it compare against the oracle itself."""
import dataclasses

import numpy as np
import pytest

import synthgen as sg
from oracle import moe, mxfp4
from oracle_pool import OracleService


@pytest.fixture(scope="module")
def svc():
    s = OracleService(n_workers=2)
    yield s
    s.close()


def test_pool_layer_and_calibration_equal_the_serial_oracle(svc):
    wl = sg.TINY
    experts = {e: moe.quantize_expert(sg.expert_w1_f32(wl, e), sg.expert_w2_f32(wl, e)) for e in range(wl.E)}
    xw = sg.activations_bf16(wl, sg.WARMUP_SEED)
    ids_w, _ = moe.topk_softmax(moe.router_logits(xw, sg.router_bf16(wl)), wl.k)
    gs1, gs2 = moe.calibrate(xw, ids_w, lambda e: experts[e], wl.swiglu_limit)
    assert svc.calibrate(wl, xw) == (gs1, gs2)
    xs = [sg.activations_bf16(wl, sg.EVAL_SEED, T=T) for T in (16, 3)]
    got = svc.layer(wl, xs, gs1, gs2)
    for x, (y, ids, w) in zip(xs, got):
        ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x, sg.router_bf16(wl)), wl.k)
        assert np.array_equal(ids, ids_ref) and np.array_equal(w, w_ref)
        assert np.array_equal(y, moe.moe_tokens(x, ids_ref, w_ref, lambda e: experts[e], gs1, gs2, wl.swiglu_limit))


def test_pool_mx_partials_equal_the_serial_oracle(svc):
    wl = dataclasses.replace(sg.TINY, name="tiny_mx_full", I=192, w_format=1)
    plan = mxfp4.tp_plan(192, 3, 32, 128)
    x = sg.activations_bf16(wl, sg.EVAL_SEED)
    ids, w = moe.topk_softmax(moe.router_logits(x, sg.router_bf16(wl)), wl.k)
    got = svc.mx_partials(wl, x, ids, [(plan, r) for r in range(3)])
    for r in range(3):
        ex = {e: mxfp4.mx_expert_shard(sg.expert_w1_f32(wl, e), sg.expert_w2_f32(wl, e), plan, r) for e in range(wl.E)}
        assert np.array_equal(got[r], mxfp4.mx_moe_partials(x, ids, lambda e: ex[e], wl.swiglu_limit))
