"""GPU: the tcgen05 block-scaled grouped GEMMs on raw operands.

Random E2M1 codes and E4M3 scales are laid out in the slot layout. Per-expert
counts are ragged, with empty experts, partial 128-row tiles and several
m-tiles, and K is partial (a stage of 2 atoms) or runs over several stages.
* W2: every real pair's fp32 row is compared with an fp64 matmul of the
  decoded operands. Padding rows must not be written.
* Cases with T >= E * 128 run the dynamic chunk schedule (prefill sizes),
  the others the static contiguous one (decode sizes).
* W1: the clamped SwiGLU + requantisation epilogue is compared with the
  oracle's quantiser applied to the fp64 reference h. Codes must agree
  except at rounding ties that the fp32 accumulation moves.
"""
import numpy as np
import pytest

from helpers import dump, ensure_built, tile_weights
from oracle import codecs, layout, moe, nvfp4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _layout(counts, seed):
    rng = np.random.default_rng(seed)
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int64)
    rng.shuffle(ids)
    return ids.reshape(-1, 1), layout.slots(ids.reshape(-1, 1), len(counts))


def _rand_operand(rng, rows, K, lo=0x30, hi=0x40):
    q = rng.integers(0, 16, (rows, K)).astype(np.uint8)
    s = rng.integers(lo, hi + 1, (rows, K // 16)).astype(np.uint8)
    return q, s


def _dec(q, s):
    R, K = q.shape
    return (codecs.e2m1_decode(q).reshape(R, K // 16, 16) * codecs.e4m3_decode(s)[:, :, None]).reshape(R, K)


def _setup(H, I, counts, seed, which):
    import torch
    from block_scaled_fp4_top_gb300 import api
    rng = np.random.default_rng(seed)
    E = len(counts)
    ids, L = _layout(counts, seed)
    T = len(ids)
    cfg = api.config(H, I, E, 1, T, 10.0)
    cap = api.capacity_rows(cfg, T)
    R = L["R"]
    K = I if which == 2 else H
    N = H if which == 2 else 2 * I
    qa, sa = _rand_operand(rng, cap, K)
    real = np.zeros(cap, dtype=bool)
    real[:R] = L["pair_of_row"] >= 0
    qa[~real] = 0
    sa[~real] = 0
    qw, sw = _rand_operand(rng, E * N, K)
    # W1 output feeds a SwiGLU clamped at 10: keep the accumulators O(1) there
    alpha = (rng.uniform(0.5, 2.0, E) * (1.0 if which == 2 else 0.25 / np.sqrt(K))).astype(np.float32)
    por = np.full(cap, -1, np.int64)
    por[:R] = L["pair_of_row"]
    dev = dict(device="cuda")
    t = dict(
        a=torch.from_numpy(nvfp4.pack_codes(qa).reshape(-1)).cuda(),
        asf=torch.from_numpy(nvfp4.swizzle(sa)).cuda(),
        w=torch.from_numpy(tile_weights(nvfp4.pack_codes(qw), N)).cuda(),
        wsf=torch.from_numpy(np.concatenate([nvfp4.swizzle(sw[e * N:(e + 1) * N]) for e in range(E)])).cuda(),
        poff=torch.from_numpy(L["padded_offsets"].astype(np.int32)).cuda(),
        por=torch.from_numpy(por.astype(np.int32)).cuda(),
        alpha=torch.from_numpy(alpha).cuda(),
        ws=torch.zeros(api.workspace_bytes(cfg), dtype=torch.uint8, **dev),
    )
    return cfg, T, cap, ids, L, (qa, sa, qw, sw, alpha), t


@pytest.mark.parametrize("H,I,counts", [
    (256, 128, [1, 0, 130, 5]),          # K = 128: one partial stage (2 scale atoms)
    (256, 768, [300, 1, 0]),             # K = 768: 3 full stages
    (512, 2048, [129, 128, 0, 2]),       # K = 2048: 8 stages around a 3-deep ring
    (256, 768, [600, 5, 130]),           # T >= E * 128: the dynamic chunk schedule (5-, 1- and 2-m-tile experts)
])
def test_w2_rows_against_fp64(H, I, counts):
    import torch
    from block_scaled_fp4_top_gb300 import api
    cfg, T, cap, ids, L, (qa, sa, qw, sw, alpha), t = _setup(H, I, counts, 1, which=2)
    o = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    api.moe_grouped_gemm_w2(cfg, T, t["a"], t["asf"], t["poff"], t["por"], t["w"], t["wsf"], t["alpha"], o, t["ws"])
    torch.cuda.synchronize()
    assert api.fp4moe_read_error(t["ws"]) == 0
    got = o.cpu().numpy()
    A = _dec(qa, sa)
    Wd = _dec(qw, sw).reshape(len(counts), H, I)
    ref = np.zeros((T, H))
    bound = np.zeros((T, H))
    for p in range(T):
        e = int(ids[p, 0])
        r = int(L["slot_of_pair"][p])
        ref[p] = alpha[e] * (Wd[e] @ A[r])
        bound[p] = alpha[e] * (np.abs(Wd[e]) @ np.abs(A[r]))
    err = np.abs(got - ref)
    ok = err <= 2e-4 * bound + 1e-30
    if not ok.all():
        dump(f"gemm_w2_{H}_{I}", got=got, ref=ref, bound=bound, qa=qa, sa=sa, qw=qw, sw=sw, alpha=alpha,
             ids=ids, slot=L["slot_of_pair"], poff=L["padded_offsets"])
    assert np.isfinite(got).all()
    assert ok.all(), f"max err/bound {(err / np.maximum(bound, 1e-30)).max():.3e}"


def test_w2_rows_to_a_16_byte_aligned_buffer():
    """A caller's o_pairs aligned to 16 bytes only gets the same rows, bit for bit, as a 32-byte-aligned one."""
    import torch
    from block_scaled_fp4_top_gb300 import api
    H, I, counts = 256, 128, [3, 0, 140]
    cfg, T, cap, ids, L, _, t = _setup(H, I, counts, 1, which=2)
    o = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    api.moe_grouped_gemm_w2(cfg, T, t["a"], t["asf"], t["poff"], t["por"], t["w"], t["wsf"], t["alpha"], o, t["ws"])
    big = torch.full((T * H + 8,), float("nan"), dtype=torch.float32, device="cuda")
    o16 = big[4:4 + T * H].view(T, H)
    assert o16.data_ptr() % 32 == 16
    api.moe_grouped_gemm_w2(cfg, T, t["a"], t["asf"], t["poff"], t["por"], t["w"], t["wsf"], t["alpha"], o16,
                            t["ws"])
    torch.cuda.synchronize()
    assert api.fp4moe_read_error(t["ws"]) == 0
    assert torch.equal(o.view(torch.int32), o16.view(torch.int32))


@pytest.mark.parametrize("H,I,counts", [(256, 128, [3, 0, 140]), (512, 256, [1, 257, 2]),
                                        (256, 128, [600, 5, 130])])   # the last one takes the dynamic schedule
def test_w1_swiglu_requant(H, I, counts):
    import torch
    from block_scaled_fp4_top_gb300 import api
    cfg, T, cap, ids, L, (qa, sa, qw, sw, alpha), t = _setup(H, I, counts, 2, which=1)
    E = len(counts)
    A = _dec(qa, sa)
    Wk = _dec(qw, sw).reshape(E, 2 * I, H)  # kernel row order
    # kernel row order -> gate/up features
    f = np.arange(I)
    gate_rows = 128 * (f // 64) + f % 64
    up_rows = gate_rows + 64
    R = L["R"]
    h = np.zeros((cap, I))
    for r in range(R):
        p = L["pair_of_row"][r]
        if p < 0:
            continue
        e = int(ids[p, 0])
        acc = Wk[e] @ A[r] * alpha[e]
        h[r] = moe.swiglu(acc[gate_rows], acc[up_rows], 10.0)
    gs2 = nvfp4.global_scale(np.float32(np.abs(h).max()))
    a2 = torch.full((cap * I // 2,), 0xEE, dtype=torch.uint8, device="cuda")
    a2sf = torch.full((cap * I // 16,), 0xEE, dtype=torch.uint8, device="cuda")
    api.moe_grouped_gemm_w1_swiglu(cfg, T, t["a"], t["asf"], t["poff"], t["por"], t["w"], t["wsf"], t["alpha"],
                                   torch.tensor([gs2], dtype=torch.float32, device="cuda"), a2, a2sf, t["ws"])
    torch.cuda.synchronize()
    assert api.fp4moe_read_error(t["ws"]) == 0
    codes = a2.cpu().numpy().reshape(cap, I // 2)[:R]
    sf = nvfp4.unswizzle(a2sf.cpu().numpy()[: R * I // 16], R, I // 16)
    q_ref, s_ref = nvfp4.quantize_rows(h[:R].astype(np.float32), gs2)
    got_deq = nvfp4.dequantize(nvfp4.unpack_codes(codes), sf, gs2)
    ref_deq = nvfp4.dequantize(q_ref, s_ref, gs2)
    real = L["pair_of_row"] >= 0           # padding rows are left untouched: compare real rows
    agree = (nvfp4.unpack_codes(codes)[real] == q_ref[real]).mean()
    if agree < 0.995:
        dump(f"gemm_w1_{H}_{I}", codes=codes, sf=sf, q_ref=q_ref, s_ref=s_ref, h=h[:R], gs2=gs2)
    assert (codes[~real] == 0xEE).all(), "padding rows must not be written"
    assert agree >= 0.995, f"code agreement {agree:.4f}"
    rel = np.linalg.norm(got_deq[real] - ref_deq[real]) / np.linalg.norm(ref_deq[real])
    assert rel < 2e-2, rel
    assert (sf[real] == s_ref[real]).mean() >= 0.99


def test_combine_reads_16_byte_aligned_rows_the_same():
    """moe_combine gives the same y, bit for bit, for pair rows in a 32-byte- and a 16-byte-aligned buffer; and
    matches the weighted sum y = bf16(sum_j w_j o_j) computed in fp64 within one bf16 rounding."""
    import torch
    from block_scaled_fp4_top_gb300 import api
    T, H, k = 37, 512, 6
    cfg = api.config(H, 128, 8, k, T, 10.0)
    g = torch.Generator(device="cuda").manual_seed(5)
    o = torch.randn(T * k, H, device="cuda", generator=g)
    w = torch.rand(T * k, device="cuda", generator=g)
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    api.moe_combine(cfg, T, o, w, y)
    big = torch.empty(T * k * H + 8, device="cuda")
    o16 = big[4:4 + T * k * H].view(T * k, H)
    o16.copy_(o)
    assert o16.data_ptr() % 32 == 16
    y16 = torch.empty_like(y)
    api.moe_combine(cfg, T, o16, w, y16)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y16.view(torch.int16))
    ref = (w.double().view(T, k, 1) * o.double().view(T, k, H)).sum(1)
    err = (y.double() - ref).abs()
    assert (err <= ref.abs() * 2.0 ** -8 + 1e-6).all()
