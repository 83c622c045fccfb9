"""Pins of the TP3 virtual-padding shard plan and the MXFP4 codec."""
import json
import os

import numpy as np

from oracle import codecs, mxfp4

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tp3_shard_plan.json")))


def test_tp3_plan_widths():
    m = GOLD["routed_moe"]
    p = mxfp4.tp_plan(m["original"], GOLD["tp"], m["align"], m["kernel_align"])
    assert p.logical_per_rank == m["logical_per_rank"] == 704
    assert p.virtual_global == m["virtual_global"] == 2112
    assert p.kernel_local == m["kernel_local"] == 768
    s = GOLD["shared_expert"]
    ps = mxfp4.tp_plan(s["original"], GOLD["tp"], s["align"], 128)
    assert (ps.logical_per_rank, ps.virtual_global) == (s["logical_per_rank"], s["virtual_global"])


def test_shard_offsets_and_tails_in_each_storage_unit():
    m = GOLD["routed_moe"]
    p = mxfp4.tp_plan(m["original"], 3, m["align"], m["kernel_align"])
    for key in ("w13_unpacked_rows", "w2_packed_bytes", "w2_e8m0_groups"):
        g = GOLD[key]
        for r in range(3):
            off, n, tail = mxfp4.shard_units(m["original"], p, r, g["unit"])
            assert off == g["source_offsets"][r], (key, r)
            assert off + n == g["source_ends"][r], (key, r)
            assert tail == g["zero_tail"][r], (key, r)
        if "unit_blind_wrong_offsets" in g:
            assert [mxfp4.shard_units(m["original"], p, r, g["unit"])[0] for r in range(3)] != g["unit_blind_wrong_offsets"]
            assert p.kernel_local // g["unit"] == g["kernel_axis"]


def test_monotonic_source_survives_shard_and_concat():
    m = GOLD["routed_moe"]
    p = mxfp4.tp_plan(m["original"], 3, m["align"], m["kernel_align"])
    for unit, width_units in [(1, 2048), (2, 1024), (32, 64)]:
        src = (np.arange(7 * width_units, dtype=np.int64) % 251 + 1).astype(np.uint8).reshape(7, width_units)
        parts = []
        for r in range(3):
            d = mxfp4.shard_axis(src, 1, m["original"], p, r, unit)
            off, n, tail = mxfp4.shard_units(m["original"], p, r, unit)
            assert d.shape[1] == p.kernel_local // unit
            assert (d[:, n:] == 0).all() and tail == d.shape[1] - n
            parts.append(d[:, :n])
        assert (np.concatenate(parts, axis=1) == src).all()


def test_mx_scale_is_floor_log2_amax_minus_2():
    v = np.zeros((4, 32), dtype=np.float32)
    v[0, 0] = 6.0        # floor(log2 6) = 2 -> X = 0 -> 6 is code 7
    v[1, 0] = 7.0        # X = 0 -> 7 saturates to 6
    v[2, 0] = 0.02       # floor(log2 0.02) = -6 -> X = -8
    v[2, 1] = -0.01
    q, s = mxfp4.mx_quantize_rows(v)
    assert list(s) == [127, 127, 127 - 8, 0]
    assert q[0, 0] == 7 and q[1, 0] == 7
    assert q[2, 0] == codecs.e2m1_encode(np.float32(0.02 * 256))  # 5.12 -> 6? nearest of {4, 6} is 6
    assert q[2, 0] == 7 and q[2, 1] == codecs.e2m1_encode(np.float32(-2.56))
    d = mxfp4.mx_dequantize(q, s)
    assert d[0, 0] == 6.0 and d[1, 0] == 6.0 and d[2, 0] == 6.0 / 256
    assert (d[3] == 0).all()
