"""GPU: the MXFP4 TP3 shard variant against the oracle.

This is the case of "Lucifer-CUTLASS TP3 virtual-padding audit": BF16
activations with MXFP4 expert weights (E2M1 codes and one E8M0 scale per 32
elements). Each rank holds a shard of logical width align_up(ceil(I / 3), 32)
inside a kernel width rounded up to 128, and everything past the logical
width is zero.

The library quantises the kernel-local fp32 shard. Its codes and scale bytes
must equal, bit for bit, those of the oracle's quantise-then-shard path. That
path cuts the full-width tensors in logical units converted to each storage
unit.

The layer's outputs must meet the float bar against the oracle's layer, and
the top-k ids must match exactly:
* at a tiny TP3 shape, on all three ranks and all tokens, with ordinary
  weights and with weights large enough that most gate and up values pass
  the SwiGLU limit;
* a NaN in one token's x gives a NaN output row, as in the oracle, and
  leaves the other tokens within the bar;
* at the DeepSeek-V4-Flash shape, all three TP3 ranks (hidden 4096, 704 of
  768, 256 experts, top-k 6) at T = 1, 8, 16 and 64, eager and under CUDA
  graph replay: each rank against the oracle's shard, and the three ranks'
  sum against the oracle's full-width layer ("4. MoE hardware tests");
* on rank 0 at T = 512, 64 sampled tokens.
The DSV4-scale oracle work runs on the test-side worker pool.
"""
import dataclasses

import numpy as np
import pytest

import synthgen as sg
from helpers import bits_to_torch, ensure_built, float_parity, torch_to_bits
from oracle import moe, mxfp4, nvfp4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def untile_mx(codes: np.ndarray, sf: np.ndarray, E: int, R: int, K: int):
    """Atom-tiled MXFP4 weights -> codes [E, R, K] and E8M0 bytes [E, R, K/32], rows in kernel order."""
    ka = K // 64
    c = codes.reshape(E, R // 128, ka, 128, 32)          # [e][row tile][atom][row][byte]
    c = c.transpose(0, 1, 3, 2, 4).reshape(E, R, ka * 32)
    q = np.empty((E, R, K), np.uint8)
    q[:, :, 0::2] = c & 0xF
    q[:, :, 1::2] = c >> 4
    s = sf.reshape(E, R // 128, ka, 128, 2).transpose(0, 1, 3, 2, 4).reshape(E, R, K // 32)
    return q, s


def kernel_to_logical_w1(q: np.ndarray, Ik: int) -> np.ndarray:
    """W1 rows from kernel order (gate/up interleaved per 64 features) back to gate rows then up rows."""
    kr = np.arange(2 * Ik)
    f = (kr // 128) * 64 + (kr % 128) % 64
    logical = np.where((kr % 128) < 64, f, Ik + f)
    out = np.empty_like(q)
    out[:, logical] = q
    return out


def shard_fp32(w1_full, w2_full, plan, rank):
    """The kernel-local fp32 shard the library quantises: logical rows / columns, zero past them."""
    I = w2_full.shape[-1]
    Ik, Il = plan.kernel_local, plan.logical_per_rank
    a, n = rank * Il, max(0, min(Il, I - rank * Il))
    w1 = np.zeros(w1_full.shape[:-2] + (2 * Ik, w1_full.shape[-1]), np.float32)
    w1[..., :n, :] = w1_full[..., a:a + n, :]
    w1[..., Ik:Ik + n, :] = w1_full[..., I + a:I + a + n, :]
    w2 = np.zeros(w2_full.shape[:-1] + (Ik,), np.float32)
    w2[..., :n] = w2_full[..., a:a + n]
    return w1, w2


def _mx_layer(H, Ik, Il, E, k, T):
    from block_scaled_fp4_top_gb300 import _lib, api
    cfg = api.config(H, Ik, E, k, T, 10.0, inter_logical=Il, w_format=_lib.W_MXFP4)
    return api.MoELayer(cfg)


def _forward(layer, x_bits, k, expect_err=0):
    import torch
    T = x_bits.shape[0]
    y = torch.empty(T, layer.cfg.hidden, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(T * k, dtype=torch.int32, device="cuda")
    layer.forward(bits_to_torch(x_bits), y, ids)
    torch.cuda.synchronize()
    assert layer.read_error() == expect_err
    return torch_to_bits(y), ids.cpu().numpy().reshape(T, k)


@pytest.mark.parametrize("w_sigma", [0.05, 1.5])   # 1.5: gate and up far past the SwiGLU limit
def test_tiny_tp3_all_ranks(w_sigma):
    import torch
    rng = np.random.default_rng(21)
    H, I, E, k, T = 256, 192, 8, 2, 16
    plan = mxfp4.tp_plan(I, 3, 32, 128)
    Ik, Il = plan.kernel_local, plan.logical_per_rank
    assert (Il, Ik) == (64, 128)
    w1f = (rng.standard_normal((E, 2 * I, H)) * w_sigma).astype(np.float32)
    w2f = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    router = moe.f32_to_bf16_bits((rng.standard_normal((E, H)) / 16).astype(np.float32))
    x_bits = moe.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x_bits, router), k)
    if w_sigma > 1:  # most gate and up values are clamped: a wrong clamp would move y far outside the bar
        gu = moe.bf16_to_f64(x_bits) @ w1f[0].astype(np.float64).T
        assert (gu[:, :I] > 10).mean() > 0.3 and (np.abs(gu[:, I:]) > 10).mean() > 0.6
    y_sum = np.zeros((T, H))
    parts = []
    for rank in range(3):
        layer = _mx_layer(H, Ik, Il, E, k, T)
        w1l, w2l = shard_fp32(w1f, w2f, plan, rank)
        layer.quantize_weights(1, 0, torch.from_numpy(w1l).cuda())
        layer.quantize_weights(2, 0, torch.from_numpy(w2l).cuda())
        layer.set_router(bits_to_torch(router))
        torch.cuda.synchronize()
        ex = {e: mxfp4.mx_expert_shard(w1f[e], w2f[e], plan, rank) for e in range(E)}
        # codes and scale bytes, bit for bit
        q1, s1 = untile_mx(layer.weights.w1_fp4.cpu().numpy(), layer.weights.w1_sf.cpu().numpy(), E, 2 * Ik, H)
        q2, s2 = untile_mx(layer.weights.w2_fp4.cpu().numpy(), layer.weights.w2_sf.cpu().numpy(), E, H, Ik)
        for e in range(E):
            assert np.array_equal(kernel_to_logical_w1(q1[e:e + 1], Ik)[0], ex[e].w1_q), (rank, e)
            assert np.array_equal(kernel_to_logical_w1(s1[e:e + 1], Ik)[0], ex[e].w1_s), (rank, e)
            assert np.array_equal(q2[e], ex[e].w2_q) and np.array_equal(s2[e], ex[e].w2_s), (rank, e)
        y, ids = _forward(layer, x_bits, k)
        assert (ids == ids_ref).all()
        y_ref = mxfp4.mx_moe_tokens(x_bits, ids_ref, w_ref, lambda e: ex[e], 10.0)
        float_parity(sg.bf16_bits_to_f32(y), sg.bf16_bits_to_f32(y_ref), bf16=True)
        y_sum += sg.bf16_bits_to_f32(y)
        parts.append(sg.bf16_bits_to_f32(y))
    # the three ranks' outputs sum to the full-width layer
    plan1 = mxfp4.tp_plan(I, 1, 32, 64)
    ex1 = {e: mxfp4.mx_expert_shard(w1f[e], w2f[e], plan1, 0) for e in range(E)}
    y_full = mxfp4.mx_moe_tokens(x_bits, ids_ref, w_ref, lambda e: ex1[e], 10.0)
    float_parity(y_sum, sg.bf16_bits_to_f32(y_full), bf16_terms=parts)


def test_nan_token_propagates_to_its_output_row():
    """bf16 activations with MXFP4 weights have no activation quantiser: a NaN in x flows through both GEMMs
    into the token's output row, as it does in the oracle. The router reports FP4MOE_ERR_EXPERT_ID for the
    token (a NaN logit ranks nowhere; it gets ids 0 with weights 0). The other tokens stay within the bar."""
    import torch
    from block_scaled_fp4_top_gb300 import _lib
    rng = np.random.default_rng(22)
    H, I, E, k, T = 256, 128, 8, 2, 16
    plan = mxfp4.tp_plan(I, 1, 32, 128)
    w1f = (rng.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)
    w2f = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    router = moe.f32_to_bf16_bits((rng.standard_normal((E, H)) / 16).astype(np.float32))
    x_bits = moe.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    x_bits[5, 40] = 0x7FC0
    layer = _mx_layer(H, I, I, E, k, T)
    layer.quantize_weights(1, 0, torch.from_numpy(w1f).cuda())
    layer.quantize_weights(2, 0, torch.from_numpy(w2f).cuda())
    layer.set_router(bits_to_torch(router))
    y, ids = _forward(layer, x_bits, k, expect_err=_lib.ERR_EXPERT_ID)
    ex = {e: mxfp4.mx_expert_shard(w1f[e], w2f[e], plan, 0) for e in range(E)}
    with np.errstate(invalid="ignore"):
        ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x_bits, router), k)
        y_ref = sg.bf16_bits_to_f32(mxfp4.mx_moe_tokens(x_bits, ids_ref, w_ref, lambda e: ex[e], 10.0))
    yf = sg.bf16_bits_to_f32(y)
    assert np.isnan(y_ref[5]).all() and np.isnan(yf[5]).all()
    others = np.arange(T) != 5
    assert (ids[others] == ids_ref[others]).all()
    float_parity(yf[others], y_ref[others], bf16=True)


def _dsv4_mx_rank_layer(wl, wl_full, plan, rank, max_tokens, chunk=8):
    """The DSV4 TP3 rank's layer: the kernel-local fp32 shard of the generator's full-width experts, cut on the
    GPU and quantised by the library."""
    import torch
    from synthgen import gpu as sgpu
    Ik, Il, If = plan.kernel_local, plan.logical_per_rank, wl_full.I
    a, n = rank * Il, max(0, min(Il, If - rank * Il))
    layer = _mx_layer(wl.H, Ik, Il, wl.E, wl.k, max_tokens)
    for e0 in range(0, wl.E, chunk):
        w1f = sgpu.expert_w1(wl_full, e0, chunk)
        w1l = torch.zeros(chunk, 2 * Ik, wl.H, dtype=torch.float32, device="cuda")
        w1l[:, :n] = w1f[:, a:a + n]
        w1l[:, Ik:Ik + n] = w1f[:, If + a:If + a + n]
        del w1f
        layer.quantize_weights(1, e0, w1l)
        w2f = sgpu.expert_w2(wl_full, e0, chunk)
        w2l = torch.zeros(chunk, wl.H, Ik, dtype=torch.float32, device="cuda")
        w2l[:, :, :n] = w2f[:, :, a:a + n]
        del w2f
        layer.quantize_weights(2, e0, w2l)
        torch.cuda.synchronize()
    layer.set_router(sgpu.router(wl))
    return layer


def test_dsv4_tp3_three_ranks_sum_to_the_full_width_layer(oracle_svc):
    import torch
    wl = sg.TP3_MXFP4
    wl_full = dataclasses.replace(wl, I=2048, I_logical=2048)   # the generator's view of the unsharded experts
    plan = mxfp4.tp_plan(2048, 3, 32, 128)
    assert (plan.logical_per_rank, plan.kernel_local) == (704, 768)
    full = mxfp4.tp_plan(2048, 1, 32, 128)
    Ts = (1, 8, 16, 64)
    x_bits = sg.activations_bf16(wl, sg.EVAL_SEED, T=max(Ts))  # the smaller batches are its leading rows
    ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x_bits, sg.router_bf16(wl)), wl.k)
    parts = oracle_svc.mx_partials(wl_full, x_bits, ids_ref, [(plan, 0), (plan, 1), (plan, 2), (full, 0)])
    y_rank_ref = [sg.bf16_bits_to_f32(moe.combine(ids_ref, w_ref, o)) for o in parts[:3]]
    y_full_ref = sg.bf16_bits_to_f32(moe.combine(ids_ref, w_ref, parts[3]))
    sums = {T: np.zeros((T, wl.H)) for T in Ts}
    parts = {T: [] for T in Ts}
    for rank in range(3):
        layer = _dsv4_mx_rank_layer(wl, wl_full, plan, rank, max(Ts))
        for T in Ts:
            y, ids = _forward(layer, x_bits[:T], wl.k)
            assert (ids == ids_ref[:T]).all(), (rank, T)
            yf = sg.bf16_bits_to_f32(y)
            float_parity(yf, y_rank_ref[rank][:T], bf16=True)
            sums[T] += yf
            parts[T].append(yf)
            # the same call captured in a CUDA graph and replayed gives the eager rows, bit for bit
            xs = bits_to_torch(x_bits[:T])
            ys = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                layer.forward(xs, ys)
            for _ in range(2):
                ys.fill_(0)
                g.replay()
                torch.cuda.synchronize()
                assert np.array_equal(torch_to_bits(ys), y), (rank, T)
            assert layer.read_error() == 0
            del g
        del layer
        torch.cuda.empty_cache()
    for T in Ts:
        float_parity(sums[T], y_full_ref[:T], bf16_terms=parts[T])


def test_dsv4_tp3_rank0_T512_sampled_tokens(oracle_svc):
    wl = sg.TP3_MXFP4
    wl_full = dataclasses.replace(wl, I=2048, I_logical=2048)
    plan = mxfp4.tp_plan(2048, 3, 32, 128)
    layer = _dsv4_mx_rank_layer(wl, wl_full, plan, 0, wl.T)
    x_bits = sg.activations_bf16(wl, sg.EVAL_SEED)
    y, ids = _forward(layer, x_bits, wl.k)
    ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x_bits, sg.router_bf16(wl)), wl.k)
    assert (ids == ids_ref).all()
    rows = np.sort(np.random.default_rng(512).choice(wl.T, 64, replace=False))
    part, = oracle_svc.mx_partials(wl_full, x_bits[rows], ids_ref[rows], [(plan, 0)])
    float_parity(sg.bf16_bits_to_f32(y[rows]), sg.bf16_bits_to_f32(moe.combine(ids_ref[rows], w_ref[rows], part)),
                 bf16=True)


def _pack_nibbles(q: np.ndarray) -> np.ndarray:
    """Codes [..., K] -> bytes [..., K / 2], element 2c in the low nibble of byte c (the checkpoint packing)."""
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("H,I,E", [(256, 192, 8), (4096, 2048, 3)])
def test_shard_mxfp4_checkpoint(H, I, E):
    """fp4moe_shard_mxfp4 cuts every TP3 rank's shard out of a full-width, already quantised MXFP4 checkpoint
    (W13 rows unpacked, W2 codes packed two per byte along I, one E8M0 byte per 32 elements). Its bytes equal
    (a) the oracle's cut of the same checkpoint, in logical units converted to each storage unit ("Packed W2
    weight is wrong", "W2 E8M0 scales are wrong"), and (b) the library's own quantisation of the rank's
    zero-padded fp32 shard. Every destination byte is written: the buffers start filled with 0xAB."""
    import torch
    rng = np.random.default_rng(31)
    w1f = (rng.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)
    w2f = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    w2f[:, 5, 32:64] = 0                                      # an all-zero group: scale byte 0 (X = -127)
    w1f[:, 7, :32] *= 1e-30                                   # a group far below the others
    cks = [mxfp4.mx_checkpoint(w1f[e], w2f[e]) for e in range(E)]
    ck13 = torch.from_numpy(np.stack([_pack_nibbles(c.w13_q) for c in cks])).cuda()
    ck13s = torch.from_numpy(np.stack([c.w13_s for c in cks])).cuda()
    ck2 = torch.from_numpy(np.stack([c.w2_packed for c in cks])).cuda()
    ck2s = torch.from_numpy(np.stack([c.w2_s for c in cks])).cuda()
    plan = mxfp4.tp_plan(I, 3, 32, 128)
    Ik, Il = plan.kernel_local, plan.logical_per_rank
    for rank in range(3):
        cut = _mx_layer(H, Ik, Il, E, 2, 16)
        for t in (cut.weights.w1_fp4, cut.weights.w1_sf, cut.weights.w2_fp4, cut.weights.w2_sf):
            t.fill_(0xAB)
        cut.shard_mxfp4_weights(1, 0, ck13, ck13s, I, 3, rank)
        cut.shard_mxfp4_weights(2, 0, ck2, ck2s, I, 3, rank)
        ref = _mx_layer(H, Ik, Il, E, 2, 16)
        w1l, w2l = shard_fp32(w1f, w2f, plan, rank)
        ref.quantize_weights(1, 0, torch.from_numpy(w1l).cuda())
        ref.quantize_weights(2, 0, torch.from_numpy(w2l).cuda())
        torch.cuda.synchronize()
        for a, b in [(cut.weights.w1_fp4, ref.weights.w1_fp4), (cut.weights.w1_sf, ref.weights.w1_sf),
                     (cut.weights.w2_fp4, ref.weights.w2_fp4), (cut.weights.w2_sf, ref.weights.w2_sf)]:
            assert torch.equal(a, b), rank
        q1, s1 = untile_mx(cut.weights.w1_fp4.cpu().numpy(), cut.weights.w1_sf.cpu().numpy(), E, 2 * Ik, H)
        q2, s2 = untile_mx(cut.weights.w2_fp4.cpu().numpy(), cut.weights.w2_sf.cpu().numpy(), E, H, Ik)
        for e in range(E):
            ex = mxfp4.mx_shard_checkpoint(cks[e], plan, rank)
            assert np.array_equal(kernel_to_logical_w1(q1[e:e + 1], Ik)[0], ex.w1_q), (rank, e)
            assert np.array_equal(kernel_to_logical_w1(s1[e:e + 1], Ik)[0], ex.w1_s), (rank, e)
            assert np.array_equal(q2[e], ex.w2_q) and np.array_equal(s2[e], ex.w2_s), (rank, e)
        del cut, ref


# ------------------------------------------ MXFP4 weights on the NVFP4 block-scaled MMA ----
#
# fp4moe_mxfp4_as_nvfp4 writes MXFP4 weights in the NVFP4 operand form: codes unchanged, each E8M0 scale
# 2^X as E4M3(2^(X - G)) on both 16-element halves, gw = 2^-G per expert matrix (G = X_max - 8). The layer
# then runs the NVFP4 hot path (NVFP4 activations). The oracle's side is mxfp4.mx_as_nvfp4 on its own MX
# shard, fed to moe's NVFP4 layer.

def _nv_layer(H, Ik, Il, E, k, T):
    from block_scaled_fp4_top_gb300 import api
    return api.MoELayer(api.config(H, Ik, E, k, T, 10.0, inter_logical=Il))


def _nv_from_mx(mx_layer, H, Ik, Il, E, k, T, e0=0):
    """An NVFP4 layer whose weights are the MXFP4 layer's, converted on the GPU; returns (layer, err word)."""
    import torch
    nv = _nv_layer(H, Ik, Il, E, k, T)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    W = mx_layer.weights
    nv.load_mxfp4_weights(1, e0, W.w1_fp4, W.w1_sf, err)
    nv.load_mxfp4_weights(2, e0, W.w2_fp4, W.w2_sf, err)
    torch.cuda.synchronize()
    return nv, err


def test_mx_as_nvfp4_bytes_match_the_oracle():
    """Codes, E4M3 scale bytes and gw of the converted weights equal mxfp4.mx_as_nvfp4 of the oracle's shard,
    on all three ranks of a tiny TP3 shape (whose zero tails are all-zero blocks)."""
    import torch
    from helpers import untile_weights
    rng = np.random.default_rng(41)
    H, I, E = 256, 192, 4
    plan = mxfp4.tp_plan(I, 3, 32, 128)
    Ik, Il = plan.kernel_local, plan.logical_per_rank
    w1f = (rng.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)
    w2f = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    w1f[:, :, :32] *= 2.0 ** -12                        # a column of blocks 12 binades down (inside the window)
    for rank in range(3):
        mx = _mx_layer(H, Ik, Il, E, 2, 16)
        w1l, w2l = shard_fp32(w1f, w2f, plan, rank)
        mx.quantize_weights(1, 0, torch.from_numpy(w1l).cuda())
        mx.quantize_weights(2, 0, torch.from_numpy(w2l).cuda())
        nv, err = _nv_from_mx(mx, H, Ik, Il, E, 2, 16)
        assert int(err[0].item()) == 0
        W = nv.weights
        for which, (codes, sf, gw) in ((1, (W.w1_fp4, W.w1_sf, W.gw1)), (2, (W.w2_fp4, W.w2_sf, W.gw2))):
            R, K = (2 * Ik, H) if which == 1 else (H, Ik)
            c = untile_weights(codes.cpu().numpy(), E * R, K // 2, R)
            s = sf.cpu().numpy().reshape(E, -1)
            for e in range(E):
                ex = mxfp4.mx_expert_shard(w1f[e], w2f[e], plan, rank)
                q, sm = (ex.w1_q, ex.w1_s) if which == 1 else (ex.w2_q, ex.w2_s)
                q_ref, sf_ref, gw_ref = mxfp4.mx_as_nvfp4(q, sm)
                got_q = nvfp4.unpack_codes(c[e * R:(e + 1) * R])
                got_s = nvfp4.unswizzle(s[e], R, K // 16)
                if which == 1:   # the NVFP4 layout keeps W1 rows in kernel order
                    got_q = kernel_to_logical_w1(got_q[None], Ik)[0]
                    got_s = kernel_to_logical_w1(got_s[None], Ik)[0]
                assert np.array_equal(got_q, q_ref), (rank, which, e)
                assert np.array_equal(got_s, sf_ref), (rank, which, e)
                assert float(gw[e].item()) == float(gw_ref), (rank, which, e)


def test_mx_as_nvfp4_flags_a_block_outside_the_window():
    """A block 20 binades below its matrix's largest has no exact E4M3 form: FP4MOE_ERR_SCALE_RANGE."""
    import torch
    from block_scaled_fp4_top_gb300 import _lib
    H, I, E = 256, 128, 2
    w1 = np.ones((E, 2 * I, H), np.float32) * 0.05
    w1[1, 3, 64:96] = 0.05 * 2.0 ** -20
    w2 = np.ones((E, H, I), np.float32) * 0.05
    mx = _mx_layer(H, I, I, E, 2, 16)
    mx.quantize_weights(1, 0, torch.from_numpy(w1).cuda())
    mx.quantize_weights(2, 0, torch.from_numpy(w2).cuda())
    _, err = _nv_from_mx(mx, H, I, I, E, 2, 16)
    assert int(err[0].item()) == _lib.ERR_SCALE_RANGE


def test_mx_weights_nvfp4_activations_tiny_tp3_ranks_sum():
    """The layer on each tiny TP3 rank against the oracle's NVFP4 layer on the NVFP4-form shard, all ranks under
    the full-width layer's activation scales; the three ranks sum to the full-width layer."""
    import torch
    rng = np.random.default_rng(43)
    H, I, E, k, T = 256, 192, 8, 2, 48
    plan = mxfp4.tp_plan(I, 3, 32, 128)
    full = mxfp4.tp_plan(I, 1, 32, 64)
    Ik, Il = plan.kernel_local, plan.logical_per_rank
    w1f = (rng.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)
    w2f = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    router = moe.f32_to_bf16_bits((rng.standard_normal((E, H)) / 16).astype(np.float32))
    x_bits = moe.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    xw_bits = moe.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))

    def nv_expert(e, pl, rank):
        ex = mxfp4.mx_expert_shard(w1f[e], w2f[e], pl, rank)
        q1, s1, g1 = mxfp4.mx_as_nvfp4(ex.w1_q, ex.w1_s)
        q2, s2, g2 = mxfp4.mx_as_nvfp4(ex.w2_q, ex.w2_s)
        return moe.QuantExpert(q1, s1, g1, q2, s2, g2)

    full_ex = {e: nv_expert(e, full, 0) for e in range(E)}
    ids_w, _ = moe.topk_softmax(moe.router_logits(xw_bits, router), k)
    gs1, gs2 = moe.calibrate(xw_bits, ids_w, lambda e: full_ex[e], 10.0)
    ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x_bits, router), k)
    y_full = sg.bf16_bits_to_f32(moe.moe_tokens(x_bits, ids_ref, w_ref, lambda e: full_ex[e], gs1, gs2, 10.0))
    parts = []
    for rank in range(3):
        mx = _mx_layer(H, Ik, Il, E, k, T)
        w1l, w2l = shard_fp32(w1f, w2f, plan, rank)
        mx.quantize_weights(1, 0, torch.from_numpy(w1l).cuda())
        mx.quantize_weights(2, 0, torch.from_numpy(w2l).cuda())
        nv, err = _nv_from_mx(mx, H, Ik, Il, E, k, T)
        assert int(err[0].item()) == 0
        nv.set_router(bits_to_torch(router))
        nv.set_global_scales(float(gs1), float(gs2))
        y, ids = _forward(nv, x_bits, k)
        assert (ids == ids_ref).all()
        ex = {e: nv_expert(e, plan, rank) for e in range(E)}
        y_ref = moe.moe_tokens(x_bits, ids_ref, w_ref, lambda e: ex[e], gs1, gs2, 10.0)
        yf = sg.bf16_bits_to_f32(y)
        float_parity(yf, sg.bf16_bits_to_f32(y_ref), bf16=True)
        parts.append(yf)
    float_parity(sum(parts), y_full, bf16_terms=parts)


def test_mx_weights_nvfp4_activations_dsv4_tp3(oracle_svc):
    """DeepSeek-V4-Flash TP3 (hidden 4096, 704 of 768, 256 experts, top-k 6) at T = 64: each rank's layer, with
    its MXFP4 shard converted on the GPU and the full-width layer's activation scales, against the oracle; the
    ranks' sum against the full-width layer; and the rank-0 layer captured in a CUDA graph replays the eager
    rows bit for bit."""
    import torch
    wl = sg.TP3_MXFP4
    wl_full = dataclasses.replace(wl, I=2048, I_logical=2048)
    plan = mxfp4.tp_plan(2048, 3, 32, 128)
    full = mxfp4.tp_plan(2048, 1, 32, 128)
    T = 64
    xw_bits = sg.activations_bf16(wl, sg.WARMUP_SEED, T=256)
    gs1, gs2 = oracle_svc.mxnv_calibrate(wl_full, xw_bits, full, 0)
    x_bits = sg.activations_bf16(wl, sg.EVAL_SEED, T=T)
    ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x_bits, sg.router_bf16(wl)), wl.k)
    parts_ref = oracle_svc.mxnv_partials(wl_full, x_bits, ids_ref, gs1, gs2,
                                         [(plan, 0), (plan, 1), (plan, 2), (full, 0)])
    y_full = sg.bf16_bits_to_f32(moe.combine(ids_ref, w_ref, parts_ref[3]))
    parts = []
    for rank in range(3):
        mx = _dsv4_mx_rank_layer(wl, wl_full, plan, rank, T)
        nv, err = _nv_from_mx(mx, wl.H, wl.I, wl.I_log, wl.E, wl.k, T)
        del mx
        assert int(err[0].item()) == 0
        nv.set_router(bits_to_torch(sg.router_bf16(wl)))
        nv.set_global_scales(float(gs1), float(gs2))
        y, ids = _forward(nv, x_bits, wl.k)
        assert (ids == ids_ref).all(), rank
        yf = sg.bf16_bits_to_f32(y)
        float_parity(yf, sg.bf16_bits_to_f32(moe.combine(ids_ref, w_ref, parts_ref[rank])), bf16=True)
        parts.append(yf)
        if rank == 0:
            xs = bits_to_torch(x_bits)
            ys = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                nv.forward(xs, ys)
            for _ in range(2):
                ys.fill_(0)
                g.replay()
                torch.cuda.synchronize()
                assert np.array_equal(torch_to_bits(ys), y)
            del g
        assert nv.read_error() == 0
        del nv
        torch.cuda.empty_cache()
    float_parity(sum(parts), y_full, bf16_terms=parts)
