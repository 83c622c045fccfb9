"""The shared seeded generator: published SplitMix64 outputs, moments, bf16 rounding."""
import numpy as np
import torch

import synthgen as sg


def test_splitmix64_reference_sequence():
    # SplitMix64 with state 1234567: the first five outputs of the reference implementation
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    s = np.array([1234567], dtype=np.uint64)
    with np.errstate(over="ignore"):
        got = [int(sg._mix64(s + np.uint64(i) * sg.GOLDEN)[0]) for i in range(1, 6)]
    assert got == want


def test_slices_are_independent_of_the_request():
    a = sg.normal_f32(7, 3, 0, 1000, 0.5)
    b = sg.normal_f32(7, 3, 400, 100, 0.5)
    assert (a[400:500] == b).all()
    assert not (sg.normal_f32(8, 3, 0, 1000, 0.5) == a).all()


def test_irwin_hall_moments():
    z = sg.normal_f32(0, 1, 0, 1 << 20, 1.0).astype(np.float64)
    assert abs(z.mean()) < 3e-3 and abs(z.std() - 1.0) < 3e-3
    assert np.abs(z).max() <= np.sqrt(3.0) * 2 + 1e-6


def test_bf16_rne_matches_torch():
    v = np.concatenate([sg.normal_f32(1, 1, 0, 100000, 3.0),
                        np.array([1.00390625, 1.01171875, -2.5e-39, 3.4e38], dtype=np.float32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (sg.f32_to_bf16_bits(v) == ref).all()


def test_zipf_bias_recipe():
    b = sg.router_bias_f32(sg.DSV4_PREFILL_ZIPF)
    assert b.shape == (256,) and (b == -1e4).sum() == 16
    live = np.sort(b[b > -1e4])[::-1]
    # p_e ~ rank^-1.1: consecutive log-probabilities differ by 1.1 * ln((r+1)/r)
    r = np.arange(1, 241)
    assert np.allclose(np.diff(live), -1.1 * np.log((r[1:]) / r[:-1]), rtol=1e-4, atol=1e-5)
