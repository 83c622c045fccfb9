"""GPU: moe_route and moe_quantize_scatter against the oracle.

Integer outputs are compared bit for bit: top-k ids, counts, offsets, padded
offsets, slot_of_pair, pair_of_row, A1 codes and swizzled scale bytes. The
router logits must agree with the oracle's exact-sum-rounded-once logits to
within one ulp. The top-k decision is taken by each side on its own fp32
logits, and that decision must be identical.
"""
import numpy as np
import pytest

import synthgen as sg
from helpers import bits_to_torch, dump, ensure_built
from oracle import layout, moe, nvfp4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def route_gpu(wl, T, x_bits, max_tokens=None):
    import torch
    from block_scaled_fp4_top_gb300 import api
    cfg = api.config(wl.H, wl.I, wl.E, wl.k, max_tokens or max(T, 1), wl.swiglu_limit)
    cap = api.capacity_rows(cfg, T)
    d = "cuda"
    i32 = dict(dtype=torch.int32, device=d)
    out = dict(logits=torch.empty(max(T, 1), wl.E, dtype=torch.float32, device=d),
               ids=torch.empty(max(T, 1) * wl.k, **i32), w=torch.empty(max(T, 1) * wl.k, dtype=torch.float32, device=d),
               counts=torch.empty(wl.E, **i32), offsets=torch.empty(wl.E, **i32), poff=torch.empty(wl.E, **i32),
               slot=torch.empty(max(T, 1) * wl.k, **i32), por=torch.full((cap,), -7, **i32))
    ws = torch.zeros(api.workspace_bytes(cfg), dtype=torch.uint8, device=d)
    x = bits_to_torch(x_bits) if T > 0 else torch.zeros(1, wl.H, dtype=torch.bfloat16, device=d)
    wr = bits_to_torch(sg.router_bf16(wl))
    bias = sg.router_bias_f32(wl)
    bias_t = None if bias is None else torch.from_numpy(bias).cuda()
    api.moe_route(cfg, T, x, wr, bias_t, out["logits"], out["ids"], out["w"], out["counts"], out["offsets"],
                  out["poff"], out["slot"], out["por"], ws)
    torch.cuda.synchronize()
    assert api.fp4moe_read_error(ws) == 0
    res = {k: v.cpu().numpy() for k, v in out.items()}
    return cfg, cap, res, x, ws


def check_route(wl, T, seed):
    x_bits = sg.activations_bf16(wl, seed, T=T)
    cfg, cap, g, _, _ = route_gpu(wl, T, x_bits)
    E, k = wl.E, wl.k
    if T == 0:
        assert (g["counts"] == 0).all() and (g["offsets"] == 0).all() and (g["poff"] == 0).all()
        return
    ref_l = moe.router_logits(x_bits, sg.router_bf16(wl), sg.router_bias_f32(wl))
    gl = g["logits"][:T]
    ulp = np.abs(gl.view(np.int32).astype(np.int64) - ref_l.view(np.int32).astype(np.int64))
    same_sign = np.signbit(gl) == np.signbit(ref_l)
    assert (same_sign | (np.abs(gl) < 1e-30)).all() and ulp.max() <= 1, f"logits differ by {ulp.max()} ulp"
    # each side decides on its own fp32 logits; the decisions must be identical
    ids_g, _ = moe.topk_softmax(gl, k)
    ids_r, w_r = moe.topk_softmax(ref_l, k)
    assert (ids_g == ids_r).all(), "a top-k decision flips between the two sides' logits (near-tie)"
    ids = g["ids"][: T * k].reshape(T, k)
    if not (ids == ids_r).all():
        dump(f"route_{wl.name}_{T}", ids=ids, ids_ref=ids_r, logits=gl, logits_ref=ref_l)
    assert (ids == ids_r).all()
    assert np.allclose(g["w"][: T * k].reshape(T, k), w_r, rtol=3e-6, atol=1e-7)
    L = layout.slots(ids_r, E)
    assert (g["counts"] == L["counts"]).all()
    assert (g["offsets"] == L["offsets"]).all()
    assert (g["poff"] == L["padded_offsets"]).all()
    assert (g["slot"][: T * k] == L["slot_of_pair"]).all()
    R = L["R"]
    assert R <= cap
    assert (g["por"][:R] == L["pair_of_row"]).all()
    return L


@pytest.mark.parametrize("wl,T", [(sg.TINY, 16), (sg.TINY, 5), (sg.TINY, 0), (sg.DSV4_DECODE, 64),
                                  (sg.DSV4_DECODE, 1), (sg.DSV4_DECODE, 333)])
def test_route_matches_oracle(wl, T):
    check_route(wl, T, sg.EVAL_SEED)


def test_route_zipf_prefill():
    wl = sg.DSV4_PREFILL_ZIPF
    L = check_route(wl, wl.T, sg.EVAL_SEED)
    # the workload's promise: some experts above 1000 tokens, and at least 16 empty experts
    assert L["counts"].max() > 1000 and (L["counts"] == 0).sum() >= 16


@pytest.mark.parametrize("wl,T", [(sg.TINY, 16), (sg.TINY, 3), (sg.DSV4_DECODE, 64)])
def test_quantize_scatter_bit_exact(wl, T):
    import torch
    from block_scaled_fp4_top_gb300 import api
    x_bits = sg.activations_bf16(wl, sg.EVAL_SEED, T=T)
    cfg, cap, g, x, ws = route_gpu(wl, T, x_bits)
    gs1 = nvfp4.global_scale(np.abs(sg.bf16_bits_to_f32(sg.activations_bf16(wl, sg.WARMUP_SEED))).max())
    a1 = torch.full((cap * wl.H // 2,), 0xAB, dtype=torch.uint8, device="cuda")
    a1sf = torch.full((cap * wl.H // 16,), 0xCD, dtype=torch.uint8, device="cuda")
    slot = torch.from_numpy(g["slot"]).cuda()
    api.moe_quantize_scatter(cfg, T, x, torch.tensor([gs1], dtype=torch.float32, device="cuda"), slot, a1, a1sf, ws)
    torch.cuda.synchronize()
    R = int(g["poff"][-1])
    codes = a1.cpu().numpy().reshape(cap, wl.H // 2)[:R]
    sf = nvfp4.unswizzle(a1sf.cpu().numpy()[: R * wl.H // 16], R, wl.H // 16)
    xf = sg.bf16_bits_to_f32(x_bits)
    q, s = nvfp4.quantize_rows(xf, gs1)
    qp = nvfp4.pack_codes(q)
    por_r = g["por"][:R]
    real = por_r >= 0                      # padding rows are unspecified and not compared
    want_c = qp[por_r[real] // wl.k]
    want_s = s[por_r[real] // wl.k]
    if not ((codes[real] == want_c).all() and (sf[real] == want_s).all()):
        dump(f"qscatter_{wl.name}_{T}", codes=codes, sf=sf, want_c=want_c, want_s=want_s)
    assert (sf[real] == want_s).all()
    assert (codes[real] == want_c).all()
