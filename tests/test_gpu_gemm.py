"""GPU: the tcgen05 block-scaled grouped GEMMs on raw operands.

Random E2M1 codes and E4M3 scales are laid out in the slot layout. Per-expert
counts are ragged, with empty experts, partial 128-row tiles and several
m-tiles, and K is partial (a stage of 2 atoms) or runs over several stages.
* W2: every real pair's bf16 row is compared with an fp64 matmul of the
  decoded operands (fp32 accumulation bound plus half a bf16 ulp).
* Cases with T >= E * 128 run the dynamic chunk schedule (prefill sizes),
  the others the static contiguous one (decode sizes). Where K and the
  weight rows are multiples of 256 (every W1) the 128 x 256 tile kernel
  runs (gemm_wide.cu); a W2 with K an odd multiple of 128 (128, 384) runs
  the 128 x 128 kernel (gemm.cu). The sparse 64-expert cases have enough
  tiles for the static schedule's tail pool: the last three tiles per CTA
  go to whichever CTAs finish their own range first. In the 128 x 128 case
  (K = 384, one ring stage per tile) the scale copiers can run tiles ahead
  of the MMAs, which tests the barrier that guards the resident scales at
  each change of expert.
* W1: the clamped SwiGLU + requantisation epilogue is compared with the
  oracle's quantiser applied to the fp64 reference h. Codes must agree
  except at rounding ties that the fp32 accumulation moves.
* Scale bytes: the 0.5 .. 2 band, and the whole finite E4M3 range (0x00,
  the subnormals 0x01 .. 0x07, up to 0x7E = 448) on both operands.
* The clamp: a W1 case whose gate and up values reach about +-50, with codes
  equal to the oracle's wherever both gate and up are clamped, and a W1 case
  with a NaN alpha, which must raise FP4MOE_ERR_NAN and leave every other
  expert's rows as they are.
"""
import numpy as np
import pytest

from helpers import assert_sched_counters_zero, bf16_ulp, dump, ensure_built, tile_weights
from oracle import codecs, layout, moe, nvfp4

pytestmark = pytest.mark.gpu


# 16 experts, 26 pairs: the static schedule with a tile or two per CTA
SPARSE16 = [1, 0, 3, 0, 2, 5, 0, 1, 2, 0, 0, 4, 1, 0, 5, 2]
# 64 experts, 48 of them live with 1-3 pairs: with 4096 weight rows that is 768 tiles of 128 x 256 (1536 of
# 128 x 128), so the static schedule keeps its last tiles in the pool that CTAs take from once their own
# range is done
SPARSE64 = [(7 * e) % 4 for e in range(64)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _layout(counts, seed):
    rng = np.random.default_rng(seed)
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int64)
    rng.shuffle(ids)
    return ids.reshape(-1, 1), layout.slots(ids.reshape(-1, 1), len(counts))


def _rand_operand(rng, rows, K, full_range=False):
    """Random E2M1 codes and E4M3 scale bytes: 0x30 .. 0x40 (0.5 .. 2), or every finite byte 0x00 .. 0x7E with
    0x00, the subnormals 0x01 .. 0x07 and 0x7E each forced into the first blocks."""
    q = rng.integers(0, 16, (rows, K)).astype(np.uint8)
    if not full_range:
        return q, rng.integers(0x30, 0x41, (rows, K // 16)).astype(np.uint8)
    s = rng.integers(0x00, 0x7F, (rows, K // 16)).astype(np.uint8)
    special = np.array([0x00, 0x01, 0x02, 0x03, 0x04, 0x05, 0x06, 0x07, 0x7E], np.uint8)
    s.reshape(-1)[: min(s.size, 4 * special.size)] = np.tile(special, 4)[: min(s.size, 4 * special.size)]
    return q, s


def _dec(q, s):
    R, K = q.shape
    return (codecs.e2m1_decode(q).reshape(R, K // 16, 16) * codecs.e4m3_decode(s)[:, :, None]).reshape(R, K)


def _setup(H, I, counts, seed, which, full_range=False, alpha_mult=1.0):
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
    qa, sa = _rand_operand(rng, cap, K, full_range)
    real = np.zeros(cap, dtype=bool)
    real[:R] = L["pair_of_row"] >= 0
    qa[~real] = 0
    sa[~real] = 0
    qw, sw = _rand_operand(rng, E * N, K, full_range)
    # W1 output feeds a SwiGLU clamped at 10: keep the accumulators O(1) there (alpha_mult drives them past it)
    alpha = (rng.uniform(0.5, 2.0, E) * (1.0 if which == 2 else 0.25 / np.sqrt(K)) * alpha_mult).astype(np.float32)
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


@pytest.mark.parametrize("H,I,counts,full_range", [
    (256, 128, [1, 0, 130, 5], False),          # K = 128: one partial stage (2 scale atoms)
    (256, 768, [300, 1, 0], False),             # K = 768: 3 full stages
    (512, 2048, [129, 128, 0, 2], False),       # K = 2048: 8 stages around a 3-deep ring
    (256, 768, [600, 5, 130], False),           # T >= E * 128: the dynamic chunk schedule (5-, 1-, 2-m-tile experts)
    (256, 768, [3, 0, 140], True),              # every finite E4M3 scale byte, static schedule
    (256, 768, [600, 5, 130], True),            # every finite E4M3 scale byte, dynamic schedule
    (512, 256, [600, 5, 130], False),           # dynamic schedule, two 256-row weight tiles of the wide kernel
    (256, 768, SPARSE16, False),                # static schedule, K = 768
    (512, 256, SPARSE16, True),                 # the same, every finite E4M3 scale byte
    (4096, 256, SPARSE64, False),               # static schedule with its tail pool, 128 x 256 tiles
    (4096, 384, SPARSE64, False),               # the same on the 128 x 128 kernel (K = 384)
])
def test_w2_rows_against_fp64(H, I, counts, full_range):
    import torch
    from block_scaled_fp4_top_gb300 import api
    cfg, T, cap, ids, L, (qa, sa, qw, sw, alpha), t = _setup(H, I, counts, 1, which=2, full_range=full_range)
    o = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")   # bf16 pair rows
    api.moe_grouped_gemm_w2(cfg, T, t["a"], t["asf"], t["poff"], t["por"], t["w"], t["wsf"], t["alpha"], o, t["ws"])
    torch.cuda.synchronize()
    assert api.fp4moe_read_error(t["ws"]) == 0
    assert_sched_counters_zero(t["ws"])
    got = o.float().cpu().numpy().astype(np.float64)
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
    ok = err <= 2e-4 * bound + 0.5 * bf16_ulp(ref) + 1e-30   # fp32 accumulation, then one bf16 rounding
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
    o = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    api.moe_grouped_gemm_w2(cfg, T, t["a"], t["asf"], t["poff"], t["por"], t["w"], t["wsf"], t["alpha"], o, t["ws"])
    big = torch.full((T * H + 16,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o16 = big[8:8 + T * H].view(T, H)
    assert o16.data_ptr() % 32 == 16
    api.moe_grouped_gemm_w2(cfg, T, t["a"], t["asf"], t["poff"], t["por"], t["w"], t["wsf"], t["alpha"], o16,
                            t["ws"])
    torch.cuda.synchronize()
    assert api.fp4moe_read_error(t["ws"]) == 0
    assert torch.equal(o.view(torch.int16), o16.view(torch.int16))


def _w1_reference(I, ids, L, qa, sa, qw, sw, alpha, cap):
    """fp64 gate, up and the oracle's SwiGLU h [cap, I] of every real row (kernel row order -> features)."""
    E = len(alpha)
    H = qa.shape[1]
    A = _dec(qa, sa)
    Wk = _dec(qw, sw).reshape(E, 2 * I, H)
    f = np.arange(I)
    gate_rows = 128 * (f // 64) + f % 64
    up_rows = gate_rows + 64
    g = np.zeros((cap, I))
    u = np.zeros((cap, I))
    for r in range(L["R"]):
        p = L["pair_of_row"][r]
        if p < 0:
            continue
        acc = Wk[int(ids[p, 0])] @ A[r] * alpha[int(ids[p, 0])]
        g[r], u[r] = acc[gate_rows], acc[up_rows]
    return g, u, moe.swiglu(g, u, 10.0)


def _run_w1(cfg, T, cap, I, t, gs2, alpha=None):
    import torch
    from block_scaled_fp4_top_gb300 import api
    a2 = torch.full((cap * I // 2,), 0xEE, dtype=torch.uint8, device="cuda")
    a2sf = torch.full((cap * I // 16,), 0xEE, dtype=torch.uint8, device="cuda")
    api.moe_grouped_gemm_w1_swiglu(cfg, T, t["a"], t["asf"], t["poff"], t["por"], t["w"], t["wsf"],
                                   t["alpha"] if alpha is None else alpha,
                                   torch.tensor([gs2], dtype=torch.float32, device="cuda"), a2, a2sf, t["ws"])
    torch.cuda.synchronize()
    assert_sched_counters_zero(t["ws"])
    return a2.cpu().numpy().reshape(cap, I // 2), a2sf.cpu().numpy()


@pytest.mark.parametrize("H,I,counts,full_range", [(256, 128, [3, 0, 140], False), (512, 256, [1, 257, 2], False),
                                                   (256, 128, [600, 5, 130], False),  # the dynamic schedule
                                                   (256, 256, [3, 0, 140], True),     # every finite E4M3 scale byte
                                                   (256, 256, [600, 5, 130], True),
                                                   (256, 256, SPARSE16, False),       # static schedule
                                                   (512, 256, SPARSE16, True),
                                                   (256, 2048, SPARSE64, False),      # the tail pool
                                                   (512, 2048, SPARSE64, True)])      # the same, K = 512
def test_w1_swiglu_requant(H, I, counts, full_range):
    from block_scaled_fp4_top_gb300 import api
    cfg, T, cap, ids, L, (qa, sa, qw, sw, alpha), t = _setup(H, I, counts, 2, which=1, full_range=full_range)
    R = L["R"]
    _, _, h = _w1_reference(I, ids, L, qa, sa, qw, sw, alpha, cap)
    gs2 = nvfp4.global_scale(np.float32(np.abs(h).max()))
    codes, sf_all = _run_w1(cfg, T, cap, I, t, gs2)
    assert api.fp4moe_read_error(t["ws"]) == 0
    codes = codes[:R]
    sf = nvfp4.unswizzle(sf_all[: R * I // 16], R, I // 16)
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


# 32 experts, 178 pairs: the static schedule over many experts, with enough rows for a thousand doubly clamped
# elements
SPARSE32 = [9, 0, 7, 12, 0, 8, 5, 0, 11, 6, 0, 9, 7, 0, 10, 4, 8, 0, 6, 13, 0, 7, 9, 0, 5, 8, 0, 12, 6, 0, 9, 7]


# static and dynamic schedules
@pytest.mark.parametrize("counts", [[3, 0, 140, 1], [600, 5, 130, 1], SPARSE32])
def test_w1_swiglu_clamp_past_the_limit(counts):
    """Gate and up driven to an RMS of about 46 (alpha x 8): a large share of both is clamped. Where gate and up are
    both past the limit, h is +-silu(10) * 10 exactly and the codes must equal the oracle's; elsewhere they agree
    up to rounding ties. A missing lower clamp on up, a gate clamped on both sides or a wrong limit fail it."""
    from block_scaled_fp4_top_gb300 import api
    H, I = 256, 256
    cfg, T, cap, ids, L, (qa, sa, qw, sw, alpha), t = _setup(H, I, counts, 4, which=1, alpha_mult=8.0)
    R = L["R"]
    g, u, h = _w1_reference(I, ids, L, qa, sa, qw, sw, alpha, cap)
    real = L["pair_of_row"] >= 0
    gr, ur = g[:R][real], u[:R][real]
    assert (gr > 10).mean() > 0.2 and (gr < -10).mean() > 0.2, "gate not driven past the limit"
    assert (np.abs(ur) > 10).mean() > 0.4, "up not driven past the limit"
    gs2 = nvfp4.global_scale(np.float32(np.abs(h).max()))
    codes, sf_all = _run_w1(cfg, T, cap, I, t, gs2)
    assert api.fp4moe_read_error(t["ws"]) == 0
    got = nvfp4.unpack_codes(codes[:R])[real]
    q_ref, s_ref = nvfp4.quantize_rows(h[:R].astype(np.float32), gs2)
    q_ref = q_ref[real]
    both = (gr > 10) & (np.abs(ur) > 10)
    assert both.sum() > 1000
    assert np.array_equal(got[both], q_ref[both]), "codes of doubly clamped elements differ from the oracle's"
    assert (got == q_ref).mean() >= 0.995
    sf = nvfp4.unswizzle(sf_all[: R * I // 16], R, I // 16)
    assert (sf[real] == s_ref[real]).mean() >= 0.99


def test_w1_nan_alpha_sets_the_nan_bit_and_spares_other_experts():
    """A NaN alpha makes its expert's gate and up NaN. The oracle's SwiGLU gives NaN there (it has no codes for
    such rows); the epilogue must raise FP4MOE_ERR_NAN, and every other expert's codes and scales must equal
    those of a run with a finite alpha, bit for bit."""
    import torch
    from block_scaled_fp4_top_gb300 import _lib, api
    H, I, counts = 256, 128, [3, 0, 140, 5]
    cfg, T, cap, ids, L, (qa, sa, qw, sw, alpha), t = _setup(H, I, counts, 6, which=1)
    R = L["R"]
    _, _, h = _w1_reference(I, ids, L, qa, sa, qw, sw, alpha, cap)
    gs2 = nvfp4.global_scale(np.float32(np.abs(h).max()))
    clean_codes, clean_sf = _run_w1(cfg, T, cap, I, t, gs2)
    assert api.fp4moe_read_error(t["ws"]) == 0
    bad = alpha.copy()
    bad[2] = np.nan
    with np.errstate(invalid="ignore"):
        _, _, h_bad = _w1_reference(I, ids, L, qa, sa, qw, sw, bad, cap)
    nan_codes, nan_sf = _run_w1(cfg, T, cap, I, t, gs2, alpha=torch.from_numpy(bad).cuda())
    assert api.fp4moe_read_error(t["ws"]) == _lib.ERR_NAN
    por = L["pair_of_row"]
    expert_of_row = np.where(por >= 0, ids[np.maximum(por, 0), 0], -1)
    rows2 = np.nonzero(expert_of_row == 2)[0]
    others = np.nonzero((expert_of_row >= 0) & (expert_of_row != 2))[0]
    assert np.isnan(h_bad[rows2]).all() and not np.isnan(h_bad[others]).any()
    assert np.array_equal(nan_codes[others], clean_codes[others])
    C = I // 16
    sfo = lambda flat: nvfp4.unswizzle(flat[: R * C], R, C)[others]
    assert np.array_equal(sfo(nan_sf), sfo(clean_sf))


def test_combine_reads_16_byte_aligned_rows_the_same():
    """moe_combine gives the same y, bit for bit, for pair rows in a 32-byte- and a 16-byte-aligned buffer; and
    matches the weighted sum y = bf16(sum_j w_j o_j) computed in fp64 within one bf16 rounding."""
    import torch
    from block_scaled_fp4_top_gb300 import api
    T, H, k = 37, 512, 6
    cfg = api.config(H, 128, 8, k, T, 10.0)
    g = torch.Generator(device="cuda").manual_seed(5)
    o = torch.randn(T * k, H, device="cuda", generator=g).bfloat16()    # bf16 pair rows
    w = torch.rand(T * k, device="cuda", generator=g)
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    api.moe_combine(cfg, T, o, w, y)
    big = torch.empty(T * k * H + 16, dtype=torch.bfloat16, device="cuda")
    o16 = big[8:8 + T * k * H].view(T * k, H)
    o16.copy_(o)
    assert o16.data_ptr() % 32 == 16
    y16 = torch.empty_like(y)
    api.moe_combine(cfg, T, o16, w, y16)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y16.view(torch.int16))
    ref = (w.double().view(T, k, 1) * o.double().view(T, k, H)).sum(1)
    err = (y.double() - ref).abs()
    assert (err <= ref.abs() * 2.0 ** -8 + 1e-6).all()
