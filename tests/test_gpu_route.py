"""GPU: moe_route and moe_quantize_scatter against the oracle.

Integer outputs are compared bit for bit: top-k ids, counts, offsets, padded
offsets, slot_of_pair, pair_of_row, A1 codes and swizzled scale bytes.

The router logits come in two passes: a tensor-core approximation l~ with the
bound d = 2^-12 |x_t| |w_e| + 2^-21 |l~|, then the exact sum rounded once for
every expert that can still reach the top k. So the logits of the selected
experts must agree with the oracle's exact-sum-rounded-once logits to within
one ulp, and every other logit must lie within its bound. The tests hold the
approximation to a quarter of the bound's first term, to check the fourfold
margin that the bound keeps over the tensor-core accumulation model. The
top-k decision is taken by each side on its own fp32 logits, and that
decision must be identical.
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


def route_gpu(wl, T, x_bits, max_tokens=None, wr_bits=None, expect_err=0):
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
    wr = bits_to_torch(sg.router_bf16(wl) if wr_bits is None else wr_bits)
    bias = sg.router_bias_f32(wl)
    bias_t = None if bias is None else torch.from_numpy(bias).cuda()
    api.moe_route(cfg, T, x, wr, bias_t, out["logits"], out["ids"], out["w"], out["counts"], out["offsets"],
                  out["poff"], out["slot"], out["por"], ws)
    torch.cuda.synchronize()
    assert api.fp4moe_read_error(ws) == expect_err
    res = {k: v.cpu().numpy() for k, v in out.items()}
    return cfg, cap, res, x, ws


def check_route(wl, T, seed):
    x_bits = sg.activations_bf16(wl, seed, T=T)
    cfg, cap, g, _, _ = route_gpu(wl, T, x_bits)
    E, k = wl.E, wl.k
    if T == 0:
        assert (g["counts"] == 0).all() and (g["offsets"] == 0).all() and (g["poff"] == 0).all()
        return
    wr_bits = sg.router_bf16(wl)
    ref_l = moe.router_logits(x_bits, wr_bits, sg.router_bias_f32(wl))
    gl = g["logits"][:T]
    ids_r, w_r = moe.topk_softmax(ref_l, k)
    # selected experts: the exact logit, to within one ulp
    sel_g = np.take_along_axis(gl, ids_r, axis=1)
    sel_r = np.take_along_axis(ref_l, ids_r, axis=1)
    ulp = np.abs(sel_g.view(np.int32).astype(np.int64) - sel_r.view(np.int32).astype(np.int64))
    same_sign = np.signbit(sel_g) == np.signbit(sel_r)
    assert (same_sign | (np.abs(sel_g) < 1e-30)).all() and ulp.max() <= 1, f"logits differ by {ulp.max()} ulp"
    # every logit: within a quarter of the pass-1 bound (plus an ulp for the exact ones)
    nx = np.sqrt((sg.bf16_bits_to_f32(x_bits).astype(np.float64) ** 2).sum(1))
    nw = np.sqrt((sg.bf16_bits_to_f32(wr_bits).astype(np.float64) ** 2).sum(1))
    quarter = 2.0 ** -14 * nx[:, None] * nw[None, :] + 2.0 ** -21 * np.abs(ref_l) + np.spacing(np.abs(ref_l))
    dev = np.abs(gl.astype(np.float64) - ref_l.astype(np.float64))
    assert (dev <= quarter).all(), f"approximate logit off by {(dev / quarter).max():.3f} of a quarter bound"
    # each side decides on its own fp32 logits; the decisions must be identical
    ids_g, _ = moe.topk_softmax(gl, k)
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
                                  (sg.DSV4_DECODE, 1), (sg.DSV4_DECODE, 333), (sg.DSV4_DECODE, 129),
                                  (sg.DSV4_DECODE, 600), (sg.TINY, 700)])
def test_route_matches_oracle(wl, T):
    check_route(wl, T, sg.EVAL_SEED)


def test_route_zipf_prefill():
    wl = sg.DSV4_PREFILL_ZIPF
    L = check_route(wl, wl.T, sg.EVAL_SEED)
    # the workload's promise: some experts above 1000 tokens, and at least 16 empty experts
    assert L["counts"].max() > 1000 and (L["counts"] == 0).sum() >= 16


# DSV4 at T = 300 and the Zipf prefill at T = 8192 take the four-blocks-per-thread path (T * H / 16 >= 65536)
@pytest.mark.parametrize("wl,T", [(sg.TINY, 16), (sg.TINY, 3), (sg.DSV4_DECODE, 64), (sg.DSV4_DECODE, 300),
                                  (sg.DSV4_PREFILL_ZIPF, 8192)])
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


@pytest.mark.parametrize("T", [40, 4100])  # one CTA per token; one warp per token from 4096 tokens on
def test_route_ties_and_zero_rows(T):
    """Exact ties: experts 3 and 5 share a router row, and token 2 is all zeros (every logit 0).
    Ties go to the lower expert id, and a zero row picks experts 0..k-1 with equal weights. With one warp per
    token, the tied tokens take the ranking of a few candidates and the zero row (every expert a candidate)
    the argmax passes."""
    wl = sg.DSV4_DECODE
    x_bits = sg.activations_bf16(wl, sg.EVAL_SEED, T=T).copy()
    x_bits[2] = 0
    wr_bits = sg.router_bf16(wl).copy()
    wr_bits[5] = wr_bits[3]
    # make 3 and 5 the favourite pair for a few tokens, so the tie sits at the top-k boundary or inside it
    x_bits[7] = wr_bits[3]
    x_bits[9] = wr_bits[3]
    _, _, g, _, _ = route_gpu(wl, T, x_bits, wr_bits=wr_bits)
    ref_l = moe.router_logits(x_bits, wr_bits, None)
    ids_r, w_r = moe.topk_softmax(ref_l, wl.k)
    ids = g["ids"][: T * wl.k].reshape(T, wl.k)
    assert (ids == ids_r).all()
    assert (ids[2] == np.arange(wl.k)).all()
    assert list(ids[7][:2]) == [3, 5] and list(ids[9][:2]) == [3, 5]
    assert np.allclose(g["w"][: T * wl.k].reshape(T, wl.k), w_r, rtol=3e-6, atol=1e-7)
    L = layout.slots(ids_r, wl.E)
    assert (g["slot"][: T * wl.k] == L["slot_of_pair"]).all()


BF16_NAN = 0x7FC0


@pytest.mark.parametrize("T", [40, 4100])  # one CTA per token; one warp per token from 4096 tokens on
def test_route_nan_router_row_is_never_picked(T):
    """A NaN logit ranks below every number: expert 11's router row holds a NaN, token 3 is expert 11's own
    row (so 11 would top its list), and no token picks 11. Everything else matches the oracle."""
    wl = sg.DSV4_DECODE
    wr_clean = sg.router_bf16(wl)
    wr_bits = wr_clean.copy()
    wr_bits[11, 5] = BF16_NAN
    x_bits = sg.activations_bf16(wl, sg.EVAL_SEED, T=T).copy()
    x_bits[3] = wr_clean[11]
    _, _, g, _, _ = route_gpu(wl, T, x_bits, wr_bits=wr_bits)
    ref_l = moe.router_logits(x_bits, wr_bits, sg.router_bias_f32(wl))
    assert np.isnan(ref_l[:, 11]).all() and np.isnan(g["logits"][:T, 11]).all()
    ids_r, w_r = moe.topk_softmax(ref_l, wl.k)
    ids = g["ids"][: T * wl.k].reshape(T, wl.k)
    assert (ids == ids_r).all() and not (ids == 11).any()
    assert np.allclose(g["w"][: T * wl.k].reshape(T, wl.k), w_r, rtol=3e-6, atol=1e-7)
    L = layout.slots(ids_r, wl.E)
    assert (g["counts"] == L["counts"]).all() and (g["slot"][: T * wl.k] == L["slot_of_pair"]).all()


@pytest.mark.parametrize("T", [40, 4100])
def test_route_nan_token_reports_expert_id_error(T):
    """A token with a NaN in its row has no comparable logit: the call reports FP4MOE_ERR_EXPERT_ID and
    that token gets ids 0 and weights 0, while every other token still matches the oracle."""
    from block_scaled_fp4_top_gb300 import _lib
    wl = sg.DSV4_DECODE
    x_bits = sg.activations_bf16(wl, sg.EVAL_SEED, T=T).copy()
    x_bits[5, 17] = BF16_NAN
    _, _, g, _, _ = route_gpu(wl, T, x_bits, expect_err=_lib.ERR_EXPERT_ID)
    ids = g["ids"][: T * wl.k].reshape(T, wl.k)
    w = g["w"][: T * wl.k].reshape(T, wl.k)
    assert (ids[5] == 0).all() and (w[5] == 0).all()
    keep = np.arange(T) != 5
    ref_l = moe.router_logits(x_bits[keep], sg.router_bf16(wl), sg.router_bias_f32(wl))
    ids_r, w_r = moe.topk_softmax(ref_l, wl.k)
    assert (ids[keep] == ids_r).all()
    assert np.allclose(w[keep], w_r, rtol=3e-6, atol=1e-7)
