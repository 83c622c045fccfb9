"""GPU: the block-FP8 shared expert against the oracle.

DeepSeek-V4-Flash has one shared expert of intermediate 2048 with block-FP8
weights and scales ("Lucifer-CUTLASS TP3 virtual-padding audit", "TP3 shape
plan" and "Paths that already appear compatible"). It runs in the same step as
the router and the routed experts ("DSV4 -> vLLM: CUDA-Graph Safety",
Graph B).

Checks:
* weight codes and fp32 block scales bit-exact against the oracle, at the
  DeepSeek-V4-Flash size and on planted blocks (all zero, an amax whose scale
  underflows, saturation, -0);
* activation codes and scales bit-exact (read from the workspace);
* o_shared within the float bar on every token of a shape with two 128-token
  tiles and a ragged tail, and at the DeepSeek-V4-Flash decode shape;
* the whole layer (routed + shared, one combine) within the float bar;
* the TP3 shards (768 features each, 768/768/512 real) against the oracle,
  and their sum against the full-width expert;
* a CUDA graph of the layer with the shared expert replays bit-identical to
  the eager call.
"""
import numpy as np
import pytest

import synthgen as sg
from helpers import OracleExperts, bits_to_torch, ensure_built, float_parity, make_layer, torch_to_bits
from oracle import codecs, fp8block, moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def w1_kernel_to_logical(q: np.ndarray, Is: int) -> np.ndarray:
    """W1 codes from kernel row order (gate and up interleaved per 64 features) back to gate rows then up rows."""
    kr = np.arange(2 * Is)
    f = (kr // 128) * 64 + kr % 64
    logical = np.where(kr % 128 < 64, f, Is + f)
    out = np.empty_like(q)
    out[logical] = q
    return out


def shared_cfg(wl, max_tokens, shared_inter=None):
    from block_scaled_fp4_top_gb300 import api
    return api.config(wl.H, wl.I, wl.E, wl.k, max_tokens, wl.swiglu_limit,
                      shared_inter=wl.shared_I if shared_inter is None else shared_inter)


def gpu_shared_weights(cfg, w1: np.ndarray | None, w2: np.ndarray | None, w1_t=None, w2_t=None):
    import torch
    from block_scaled_fp4_top_gb300 import api
    b = api.shared_weight_bytes(cfg)
    se = api.SharedWeights(torch.empty(b[0], dtype=torch.uint8, device="cuda"),
                           torch.empty(b[1] // 4, dtype=torch.float32, device="cuda"),
                           torch.empty(b[2], dtype=torch.uint8, device="cuda"),
                           torch.empty(b[3] // 4, dtype=torch.float32, device="cuda"))
    w1_t = torch.from_numpy(w1).cuda() if w1_t is None else w1_t
    w2_t = torch.from_numpy(w2).cuda() if w2_t is None else w2_t
    api.fp4moe_shared_quantize_weights(cfg, 1, w1_t, se.w1, se.w1_scales)
    api.fp4moe_shared_quantize_weights(cfg, 2, w2_t, se.w2, se.w2_scales)
    torch.cuda.synchronize()
    return se


def gpu_o_shared(cfg, se, x_bits):
    import torch
    from block_scaled_fp4_top_gb300 import api
    T = x_bits.shape[0]
    ws = torch.zeros(api.workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    o = torch.full((max(T, 1), cfg.hidden), float("nan"), dtype=torch.float32, device="cuda")
    api.moe_shared_expert(cfg, T, bits_to_torch(x_bits), se, o, ws)
    torch.cuda.synchronize()
    assert api.fp4moe_read_error(ws) == 0
    return o[:T].cpu().numpy().astype(np.float64), ws


def check_weights(cfg, se, w1, w2):
    Is, H = cfg.shared_inter, cfg.hidden
    q1 = w1_kernel_to_logical(se.w1.cpu().numpy().reshape(2 * Is, H), Is)
    s1 = se.w1_scales.cpu().numpy().reshape(2 * Is // 128, H // 128)         # logical block order
    q1_ref, s1_ref = fp8block.quantize_blocks(w1)
    assert (s1.view(np.uint32) == s1_ref.view(np.uint32)).all(), f"{(s1 != s1_ref).sum()} W1 scales differ"
    assert (q1 == q1_ref).all(), f"{(q1 != q1_ref).sum()} W1 codes differ"
    q2_ref, s2_ref = fp8block.quantize_blocks(w2)
    assert (se.w2_scales.cpu().numpy().reshape(H // 128, Is // 128).view(np.uint32) == s2_ref.view(np.uint32)).all()
    assert (se.w2.cpu().numpy().reshape(H, Is) == q2_ref).all()


def test_weights_bit_exact_dsv4_size():
    wl = sg.DSV4_DECODE_SHARED
    cfg = shared_cfg(wl, 64)
    w1, w2 = sg.shared_w1_f32(wl), sg.shared_w2_f32(wl)
    check_weights(cfg, gpu_shared_weights(cfg, w1, w2), w1, w2)


def test_weights_bit_exact_planted_blocks():
    rng = np.random.default_rng(23)
    H, Is = 512, 256
    cfg = shared_cfg(sg.TINY, 16, shared_inter=Is)
    cfg.hidden = H
    w1 = (rng.standard_normal((2 * Is, H)) * 0.02).astype(np.float32)
    w2 = (rng.standard_normal((H, Is)) * 0.02).astype(np.float32)
    w1[0:128, 0:128] = 0.0                                       # all-zero block: scale 0, codes 0
    w1[128:256, 128:256] = 0.0
    w1[200, 200] = np.float32(2.0 ** -149)                       # amax / 448 underflows to 0
    w1[300:428, 256:384] *= np.float32(1e30)                     # large magnitudes, still finite scales
    w2[5, :] = -0.0                                              # negative zeros keep their sign code 0x80
    w2[5, 0] = np.float32(-1e-3)
    check_weights(cfg, gpu_shared_weights(cfg, w1, w2), w1, w2)


def test_activation_codes_bit_exact_and_o_shared_all_tokens():
    from block_scaled_fp4_top_gb300 import api
    wl = sg.TINY_SHARED                                          # T = 200: two 128-token tiles, ragged tail
    cfg = shared_cfg(wl, wl.T)
    w1, w2 = sg.shared_w1_f32(wl), sg.shared_w2_f32(wl)
    se = gpu_shared_weights(cfg, w1, w2)
    x = sg.activations_bf16(wl, sg.EVAL_SEED)
    o, ws = gpu_o_shared(cfg, se, x)
    # the activation codes and scales sit after the routed regions of the workspace: [tcap][H] codes, then
    # [H/128][tcap] scales, each region 256-byte aligned
    base = api.workspace_bytes(shared_cfg(wl, wl.T, shared_inter=0))
    tcap = 256
    wsn = ws.cpu().numpy()
    qx = wsn[base:base + tcap * wl.H].reshape(tcap, wl.H)[:wl.T]
    off = base + (tcap * wl.H + 255) // 256 * 256
    sx = wsn[off:off + 4 * tcap * (wl.H // 128)].view(np.float32).reshape(wl.H // 128, tcap)[:, :wl.T].T
    q_ref, s_ref = fp8block.quantize_groups(moe.bf16_to_f64(x).astype(np.float32))
    assert (sx.view(np.uint32) == s_ref.view(np.uint32)).all()
    assert (qx == q_ref).all(), f"{(qx != q_ref).sum()} activation codes differ"
    ref = fp8block.shared_out(x, fp8block.quantize_shared(w1, w2), wl.swiglu_limit)
    float_parity(o, ref)


def test_o_shared_dsv4_decode_all_tokens():
    wl = sg.DSV4_DECODE_SHARED
    cfg = shared_cfg(wl, wl.T)
    w1, w2 = sg.shared_w1_f32(wl), sg.shared_w2_f32(wl)
    se = gpu_shared_weights(cfg, w1, w2)
    x = sg.activations_bf16(wl, sg.EVAL_SEED)
    o, _ = gpu_o_shared(cfg, se, x)
    float_parity(o, fp8block.shared_out(x, fp8block.quantize_shared(w1, w2), wl.swiglu_limit))


def test_o_shared_dsv4_ragged_prefill_sampled_rows():
    wl = sg.DSV4_DECODE_SHARED
    T = 1000                                                     # eight 128-token tiles, the last holds 104
    cfg = shared_cfg(wl, T)
    w1, w2 = sg.shared_w1_f32(wl), sg.shared_w2_f32(wl)
    se = gpu_shared_weights(cfg, w1, w2)
    x = sg.activations_bf16(wl, sg.EVAL_SEED, T=T)
    o, _ = gpu_o_shared(cfg, se, x)
    rows = np.array([0, 127, 128, 511, 895, 896, 999])
    float_parity(o[rows], fp8block.shared_out(x[rows], fp8block.quantize_shared(w1, w2), wl.swiglu_limit))


def layer_with_shared(wl, max_tokens):
    from synthgen import gpu as sgpu
    from block_scaled_fp4_top_gb300 import api
    import torch
    base = make_layer(wl, max_tokens)                            # routed weights from the generator
    cfg = shared_cfg(wl, max_tokens)
    layer = api.MoELayer(cfg)
    layer.weights = base.weights
    layer.router_w, layer.router_bias = base.router_w, base.router_bias
    layer.quantize_shared_weights(1, sgpu.shared_w1(wl))
    layer.quantize_shared_weights(2, sgpu.shared_w2(wl))
    torch.cuda.synchronize()
    return layer


def test_layer_with_shared_expert_tiny_all_tokens():
    wl = sg.TINY_SHARED
    layer = layer_with_shared(wl, wl.T)
    layer.calibrate(bits_to_torch(sg.activations_bf16(wl, sg.WARMUP_SEED)))
    gs1, gs2 = np.float32(layer.gs1.item()), np.float32(layer.gs2.item())
    x = sg.activations_bf16(wl, sg.EVAL_SEED)
    import torch
    y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(wl.T * wl.k, dtype=torch.int32, device="cuda")
    layer.forward(bits_to_torch(x), y, ids)
    torch.cuda.synchronize()
    assert layer.read_error() == 0
    ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x, sg.router_bf16(wl), None), wl.k)
    assert (ids.cpu().numpy().reshape(wl.T, wl.k) == ids_ref).all()
    o_ref = fp8block.shared_out(x, fp8block.quantize_shared(sg.shared_w1_f32(wl), sg.shared_w2_f32(wl)),
                                wl.swiglu_limit)
    y_ref = moe.moe_tokens(x, ids_ref, w_ref, OracleExperts(wl), gs1, gs2, wl.swiglu_limit, shared=o_ref)
    float_parity(sg.bf16_bits_to_f32(torch_to_bits(y)), sg.bf16_bits_to_f32(y_ref), bf16=True)


def test_layer_with_shared_expert_dsv4_decode_and_graph_replay():
    import torch
    from synthgen import gpu as sgpu
    wl = sg.DSV4_DECODE_SHARED
    layer = layer_with_shared(wl, wl.T)
    layer.calibrate(bits_to_torch(sg.activations_bf16(wl, sg.WARMUP_SEED)))
    gs1, gs2 = np.float32(layer.gs1.item()), np.float32(layer.gs2.item())
    x = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    y_e = torch.empty_like(x)
    ids = torch.empty(wl.T * wl.k, dtype=torch.int32, device="cuda")
    sgpu.activations(wl, sg.EVAL_SEED, out=x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x, y, ids)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, y, ids)
    for i in range(3):
        sgpu.activations(wl, sg.REPLAY_SEED0 + i, out=x)
        g.replay()
        layer.forward(x, y_e, None)
        assert torch.equal(y, y_e), f"replay {i}: graph and eager differ"
    torch.cuda.synchronize()
    assert layer.read_error() == 0
    # the last replay's sampled rows against the oracle
    x_bits = sg.activations_bf16(wl, sg.REPLAY_SEED0 + 2)
    ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x_bits, sg.router_bf16(wl), None), wl.k)
    assert (ids.cpu().numpy().reshape(wl.T, wl.k) == ids_ref).all()
    rows = np.array([0, 33, 63])
    o_ref = fp8block.shared_out(x_bits[rows], fp8block.quantize_shared(sg.shared_w1_f32(wl), sg.shared_w2_f32(wl)),
                                wl.swiglu_limit)
    y_ref = moe.moe_tokens(x_bits[rows], ids_ref[rows], w_ref[rows], OracleExperts(wl), gs1, gs2, wl.swiglu_limit,
                           shared=o_ref)
    float_parity(sg.bf16_bits_to_f32(torch_to_bits(y)[rows]), sg.bf16_bits_to_f32(y_ref), bf16=True)


def test_tp3_shards_against_oracle_and_their_sum():
    rng = np.random.default_rng(29)
    H, I, T = 256, 2048, 64
    w1 = (rng.standard_normal((2 * I, H)) * 0.02).astype(np.float32)
    w2 = (rng.standard_normal((H, I)) * 0.02).astype(np.float32)
    x = moe.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    total = np.zeros((T, H))
    for r in range(3):
        s1, s2 = fp8block.tp_shard(w1, w2, r, 3)
        cfg = shared_cfg(sg.TINY, T, shared_inter=768)
        cfg.hidden = H
        o, _ = gpu_o_shared(cfg, gpu_shared_weights(cfg, s1, s2), x)
        float_parity(o, fp8block.shared_out(x, fp8block.quantize_shared(s1, s2), 10.0))
        total += o
    cfg = shared_cfg(sg.TINY, T, shared_inter=I)
    cfg.hidden = H
    full, _ = gpu_o_shared(cfg, gpu_shared_weights(cfg, w1, w2), x)
    float_parity(total, full, rel_l2=1e-4, max_abs_rms=1e-3)
