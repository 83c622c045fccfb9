"""GPU: the generator twin equals the numpy generator, and the device NVFP4
block quantiser equals the oracle's bit for bit (codes and scale bytes)."""
import numpy as np
import pytest

import synthgen as sg
from helpers import bits_to_torch, dump, ensure_built, torch_to_bits
from oracle import codecs, nvfp4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_generator_twin_matches_numpy():
    import torch
    from synthgen import gpu as sgpu
    wl = sg.DSV4_DECODE
    x = sgpu.activations(wl, 5, T=8)
    assert (torch_to_bits(x) == sg.activations_bf16(wl, 5, T=8)).all()
    w1 = sgpu.expert_w1(sg.TINY, 3, 2)
    ref = np.stack([sg.expert_w1_f32(sg.TINY, 3), sg.expert_w1_f32(sg.TINY, 4)])
    assert (w1.cpu().numpy().view(np.uint32) == ref.view(np.uint32)).all()
    assert (torch_to_bits(sgpu.router(sg.TINY)) == sg.router_bf16(sg.TINY)).all()
    w2 = sgpu.expert_w2(wl, 255, 1)
    assert (w2.cpu().numpy()[0] == sg.expert_w2_f32(wl, 255)).all()
    se = sg.TINY_SHARED
    assert (sgpu.shared_w1(se).cpu().numpy().view(np.uint32) == sg.shared_w1_f32(se).view(np.uint32)).all()
    assert (sgpu.shared_w2(se).cpu().numpy().view(np.uint32) == sg.shared_w2_f32(se).view(np.uint32)).all()
    torch.cuda.synchronize()


def quant_rows_gpu(v: np.ndarray, g: np.ndarray):
    import torch
    from block_scaled_fp4_top_gb300 import api
    R, K = v.shape
    codes = torch.empty(R * K // 2, dtype=torch.uint8, device="cuda")
    sf = torch.empty(R * K // 16, dtype=torch.uint8, device="cuda")
    api.fp4moe_quantize_rows_f32(R, K, torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda(),
                                 torch.from_numpy(np.ascontiguousarray(g, np.float32)).cuda(), codes, sf)
    return codes.cpu().numpy().reshape(R, K // 2), nvfp4.unswizzle(sf.cpu().numpy(), R, K // 16)


def check_against_oracle(v, g, name):
    codes, sf = quant_rows_gpu(v, g)
    q_ref, sf_ref = nvfp4.quantize_rows(v, g)
    ok_sf = (sf == sf_ref)
    ok_codes = (codes == nvfp4.pack_codes(q_ref))
    if not (ok_sf.all() and ok_codes.all()):
        dump(name, v=v, g=g, codes=codes, sf=sf, codes_ref=nvfp4.pack_codes(q_ref), sf_ref=sf_ref)
    assert ok_sf.all(), f"{(~ok_sf).sum()} scale bytes differ"
    assert ok_codes.all(), f"{(~ok_codes).sum()} code bytes differ"


def test_random_rows_bit_exact():
    rng = np.random.default_rng(0)
    R, K = 256, 512
    v = (rng.standard_normal((R, K)) * np.exp(rng.uniform(-8, 8, (R, 1)))).astype(np.float32)
    v[::7, ::5] = 0.0
    v[3, :] = -0.0
    g = nvfp4.global_scale(np.abs(v).max()) * np.exp(rng.uniform(-3, 3, R)).astype(np.float32)
    check_against_oracle(v, g.astype(np.float32), "quant_random")


def _sweep(mags):
    m = np.array(mags, dtype=np.float64)
    pts = list(m) + list(0.5 * (m[:-1] + m[1:]))
    out = []
    for p in pts:
        p32 = np.float32(p)
        out += [p32, np.nextafter(p32, np.float32(np.inf)), np.nextafter(p32, np.float32(0))]
    return np.array(out, dtype=np.float32)


def test_e2m1_rounding_of_every_boundary():
    # amax 6 and g = 1 give s = 1, sf = 1.0 and inv = 1, so each code is E2M1(v)
    vals = _sweep(list(codecs.E2M1_MAGS) + [8.0])
    vals = np.concatenate([vals, -vals, [np.float32(-0.0), np.float32(-1e-20)]]).astype(np.float32)
    vals = np.clip(vals, -6, 6)
    per = 15
    nb = (len(vals) + per - 1) // per
    blocks = np.zeros((nb, 16), dtype=np.float32)
    blocks[:, 0] = 6.0
    flat = np.zeros(nb * per, dtype=np.float32)
    flat[: len(vals)] = vals
    blocks[:, 1:] = flat.reshape(nb, per)
    K = 64
    rows = (nb * 16 + K - 1) // K
    R = (rows + 127) // 128 * 128
    v = np.zeros((R, K), dtype=np.float32)
    v.reshape(-1)[: nb * 16] = blocks.reshape(-1)
    check_against_oracle(v, np.ones(R, np.float32), "quant_e2m1_sweep")


def test_e4m3_scale_rounding_sweep():
    # amax 6 gives s = g, so each scale byte is E4M3(g): sweep g over every E4M3 boundary
    gs = _sweep(list(codecs.E4M3_MAGS[1:]) + [480.0])
    gs = np.concatenate([gs, np.float32([1e-12, 2.0**-10, 3e-3, 500.0, 1e6])]).astype(np.float32)
    R = (len(gs) + 127) // 128 * 128
    g = np.ones(R, np.float32)
    g[: len(gs)] = gs
    v = np.zeros((R, 64), dtype=np.float32)
    v[:, 0] = 6.0
    v[:, 1] = 1.5
    v[:, 17] = -3.0
    check_against_oracle(v, g, "quant_e4m3_sweep")
