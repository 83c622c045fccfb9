"""The C ABI library on the CPU: it loads, exports every symbol declared in
include/fp4moe.h, and its host-side argument checks and sizing are right.
No call here reaches a CUDA API: every checked call fails validation first."""
import ctypes
import os
import re

import pytest

from helpers import ROOT, ensure_built
from oracle import layout


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    from block_scaled_fp4_top_gb300 import _lib
    return _lib.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "fp4moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s+\*?([a-z_0-9]+)\s*\(", src, flags=re.M))


def test_every_declared_symbol_is_exported(lib):
    from block_scaled_fp4_top_gb300 import _lib
    names = header_functions()
    assert "moe_forward" in names and "moe_route" in names and len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(_lib.SIGNATURES), names ^ set(_lib.SIGNATURES)


def test_library_does_not_link_libcuda():
    ensure_built()
    from block_scaled_fp4_top_gb300 import _lib
    import subprocess
    out = subprocess.run(["ldd", _lib.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def _cfg(**kw):
    from block_scaled_fp4_top_gb300 import api
    d = dict(hidden=4096, inter=2048, num_experts=256, top_k=6, max_tokens=64, swiglu_limit=10.0)
    d.update(kw)
    return api.config(**d)


def test_capacity_matches_oracle(lib):
    for T in [0, 1, 2, 21, 22, 64, 100, 4096, 8192]:
        for k, E in [(6, 256), (2, 8)]:
            cfg = _cfg(top_k=k, num_experts=E, max_tokens=8192)
            assert lib.fp4moe_capacity_rows(ctypes.byref(cfg), T) == layout.capacity_rows(T, k, E)


def test_sizes(lib):
    cfg = _cfg()
    from block_scaled_fp4_top_gb300 import api
    b1, s1, b2, s2 = api.weight_bytes(cfg)
    assert (b1, s1, b2, s2) == (256 * 4096 * 4096 // 2, 256 * 4096 * 4096 // 16, 256 * 4096 * 2048 // 2,
                                256 * 4096 * 2048 // 16)
    ws = api.workspace_bytes(cfg)
    cap = layout.capacity_rows(64, 6, 256)
    assert ws >= cap * (4096 // 2 + 4096 // 16 + 2048 // 2 + 2048 // 16) + 64 * 6 * 4096 * 2   # bf16 pair rows
    assert api.workspace_bytes(_cfg(hidden=100)) == 0  # unsupported shape -> 0


def test_argument_checks(lib):
    from block_scaled_fp4_top_gb300 import _lib
    cfg = _cfg()
    p = ctypes.c_void_p(0x10000)     # aligned, never dereferenced: validation fails first
    bad = ctypes.c_void_p(0x10004)
    null = None
    args = [p] * 13
    # null pointer
    assert lib.moe_route(ctypes.byref(cfg), 8, null, *args[1:]) == _lib.INVALID_ARG
    # misaligned
    assert lib.moe_route(ctypes.byref(cfg), 8, bad, *args[1:]) == _lib.MISALIGNED
    # T beyond max_tokens
    assert lib.moe_route(ctypes.byref(cfg), 65, *args) == _lib.CAPACITY
    assert lib.moe_route(ctypes.byref(cfg), -1, *args) == _lib.INVALID_ARG
    # unsupported shapes / format
    assert lib.moe_route(ctypes.byref(_cfg(hidden=4000)), 8, *args) == _lib.UNSUPPORTED
    assert lib.moe_route(ctypes.byref(_cfg(top_k=17)), 8, *args) == _lib.UNSUPPORTED
    assert lib.moe_route(ctypes.byref(_cfg(w_format=2)), 8, *args) == _lib.UNSUPPORTED          # unknown format
    # MXFP4: the logical width must be whole 32-element groups inside the kernel width
    assert lib.moe_route(ctypes.byref(_cfg(w_format=_lib.W_MXFP4, inter=768, inter_logical=800)), 8,
                         *args) == _lib.UNSUPPORTED
    assert lib.moe_route(ctypes.byref(_cfg(w_format=_lib.W_MXFP4, inter=768, inter_logical=700)), 8,
                         *args) == _lib.UNSUPPORTED
    assert lib.fp4moe_calibrate(ctypes.byref(_cfg(w_format=_lib.W_MXFP4, inter=768, inter_logical=704)), 8,
                                *([p] * 10)) == _lib.UNSUPPORTED
    assert lib.moe_forward(None, 8, *([p] * 16)) == _lib.INVALID_ARG
    assert lib.fp4moe_quantize_rows_f32(100, 64, p, p, p, p, p) == _lib.INVALID_ARG  # rows % 128
    assert lib.fp4moe_selftest_wait_timeout(p, 0, p, None) == _lib.INVALID_ARG          # limit below 1 ms
    assert lib.fp4moe_selftest_wait_timeout(p, 60_000_000, p, None) == _lib.INVALID_ARG  # above 50 ms
    assert lib.fp4moe_selftest_wait_timeout(ctypes.c_void_p(0x10002), 5_000_000, p, None) == _lib.MISALIGNED
    assert lib.fp4moe_status_string(_lib.CAPACITY) == b"FP4MOE_CAPACITY"
    assert lib.fp4moe_abi_version() == 105


def test_shared_expert_checks_and_sizes(lib):
    from block_scaled_fp4_top_gb300 import _lib, api
    p = ctypes.c_void_p(0x10000)
    cfg = _cfg(shared_inter=2048)
    assert api.shared_weight_bytes(cfg) == (2 * 2048 * 4096, 32 * 32 * 4, 4096 * 2048, 32 * 16 * 4)
    tcap = 128                                            # max_tokens 64 rounded up to whole 128-row tiles
    grow = tcap * 4096 + 32 * tcap * 4 + tcap * 2048 + 16 * tcap * 4 + 64 * 4096 * 4
    assert api.workspace_bytes(cfg) >= api.workspace_bytes(_cfg()) + grow
    # widths that are not whole 128 x 128 blocks, and negative widths
    assert lib.moe_route(ctypes.byref(_cfg(shared_inter=100)), 8, *([p] * 13)) == _lib.UNSUPPORTED
    assert lib.moe_route(ctypes.byref(_cfg(shared_inter=-128)), 8, *([p] * 13)) == _lib.INVALID_ARG
    se = _lib.SharedWeights(0x10000, 0x10000, 0x10000, 0x10000)
    se_bad = _lib.SharedWeights(0x10000, 0x10008, 0x10000, 0x10000)
    se_null = _lib.SharedWeights(0x10000, None, 0x10000, 0x10000)
    # a layer without a shared expert, a missing struct, null or misaligned members
    assert lib.moe_shared_expert(ctypes.byref(_cfg()), 8, p, ctypes.byref(se), p, p, None) == _lib.INVALID_ARG
    assert lib.moe_shared_expert(ctypes.byref(cfg), 8, p, None, p, p, None) == _lib.INVALID_ARG
    assert lib.moe_shared_expert(ctypes.byref(cfg), 8, p, ctypes.byref(se_null), p, p, None) == _lib.INVALID_ARG
    assert lib.moe_shared_expert(ctypes.byref(cfg), 8, p, ctypes.byref(se_bad), p, p, None) == _lib.MISALIGNED
    assert lib.moe_shared_expert(ctypes.byref(cfg), 65, p, ctypes.byref(se), p, p, None) == _lib.CAPACITY
    assert lib.moe_forward_shared(ctypes.byref(cfg), 8, *([p] * 11), None, *([p] * 5)) == _lib.INVALID_ARG
    assert lib.fp4moe_shared_quantize_weights(ctypes.byref(cfg), 3, p, p, p, None) == _lib.INVALID_ARG
    assert lib.fp4moe_shared_quantize_weights(ctypes.byref(_cfg()), 1, p, p, p, None) == _lib.INVALID_ARG
    # an expert-parallel combine must be told which pairs are held here
    ep = _cfg(ep_first=0, ep_count=64)
    assert lib.moe_combine_shared(ctypes.byref(ep), 8, p, p, None, p, p, None) == _lib.INVALID_ARG


def test_tp_shard_units_reproduce_the_tp3_plan(lib):
    """The library's shard plan against the offsets and zero tails that "Lucifer-CUTLASS TP3 virtual-padding
    audit" prints for 2048 over three ranks ("TP3 shape plan", "Packed W2 weight is wrong", "W2 E8M0 scales are
    wrong"), in each tensor's storage unit, and against the oracle's plan on other widths."""
    import json
    from block_scaled_fp4_top_gb300 import api
    from oracle import mxfp4
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "tp3_shard_plan.json")))
    m = g["routed_moe"]
    for key in ("w13_unpacked_rows", "w2_packed_bytes", "w2_e8m0_groups"):
        ax = g[key]
        got = [api.fp4moe_tp_shard_units(m["original"], g["tp"], m["align"], m["kernel_align"], r, ax["unit"])
               for r in range(g["tp"])]
        assert [o for o, _, _ in got] == ax["source_offsets"], key
        assert [o + n for o, n, _ in got] == ax["source_ends"], key
        assert [z for _, _, z in got] == ax["zero_tail"], key
        assert {n + z for _, n, z in got} == {m["kernel_local"] // ax["unit"]}, key
    for width, tp, unit in [(2048, 1, 32), (2048, 2, 2), (2048, 4, 32), (1536, 3, 32), (4096, 8, 2), (96, 3, 32)]:
        plan = mxfp4.tp_plan(width, tp, 32, 128)
        for r in range(tp):
            assert api.fp4moe_tp_shard_units(width, tp, 32, 128, r, unit) == mxfp4.shard_units(width, plan, r, unit)


def test_tp_shard_checks(lib):
    from block_scaled_fp4_top_gb300 import _lib
    out = [ctypes.c_int32() for _ in range(3)]
    refs = [ctypes.byref(v) for v in out]
    assert lib.fp4moe_tp_shard_units(2048, 3, 32, 128, 3, 1, *refs) == _lib.INVALID_ARG       # rank >= tp
    assert lib.fp4moe_tp_shard_units(2048, 0, 32, 128, 0, 1, *refs) == _lib.INVALID_ARG       # no ranks
    assert lib.fp4moe_tp_shard_units(2048, 3, 32, 128, 1, 3, *refs) == _lib.UNSUPPORTED       # 704 splits a unit
    assert lib.fp4moe_tp_shard_units(2048, 3, 32, 128, 2, 32, None, None, None) == _lib.OK   # outputs optional
    p = ctypes.c_void_p(0x10000)
    mx = _cfg(w_format=_lib.W_MXFP4, inter=768, inter_logical=704)
    assert lib.fp4moe_shard_mxfp4(ctypes.byref(_cfg()), 1, 4, 2048, 3, 0, p, p, p, p, None) == _lib.UNSUPPORTED
    assert lib.fp4moe_shard_mxfp4(ctypes.byref(mx), 3, 4, 2048, 3, 0, p, p, p, p, None) == _lib.INVALID_ARG
    assert lib.fp4moe_shard_mxfp4(ctypes.byref(mx), 1, 4, 2048, 2, 0, p, p, p, p, None) == _lib.INVALID_ARG  # widths
    assert lib.fp4moe_shard_mxfp4(ctypes.byref(mx), 1, 4, 2040, 3, 0, p, p, p, p, None) == _lib.UNSUPPORTED
    assert lib.fp4moe_shard_mxfp4(ctypes.byref(mx), 1, 4, 2048, 3, 3, p, p, p, p, None) == _lib.INVALID_ARG  # rank
    assert lib.fp4moe_shard_mxfp4(ctypes.byref(mx), 2, 4, 2048, 3, 1, p, None, p, p, None) == _lib.INVALID_ARG
    assert lib.fp4moe_shard_mxfp4(ctypes.byref(mx), 2, 4, 2048, 3, 1, p, p, ctypes.c_void_p(0x10008), p,
                                  None) == _lib.MISALIGNED


def test_mxfp4_as_nvfp4_and_probe_checks(lib):
    """Argument checks of the MXFP4-to-NVFP4 weight conversion and of the tensor-core probe; each fails before
    any CUDA call."""
    from block_scaled_fp4_top_gb300 import _lib
    p = ctypes.c_void_p(0x10000)
    nv = _cfg(inter=768, inter_logical=704)
    mx = _cfg(w_format=_lib.W_MXFP4, inter=768, inter_logical=704)
    assert lib.fp4moe_mxfp4_as_nvfp4(ctypes.byref(mx), 1, 4, p, p, p, p, p, p, None) == _lib.UNSUPPORTED
    assert lib.fp4moe_mxfp4_as_nvfp4(ctypes.byref(nv), 3, 4, p, p, p, p, p, p, None) == _lib.INVALID_ARG
    assert lib.fp4moe_mxfp4_as_nvfp4(ctypes.byref(nv), 1, 257, p, p, p, p, p, p, None) == _lib.INVALID_ARG
    assert lib.fp4moe_mxfp4_as_nvfp4(ctypes.byref(nv), 1, 4, p, p, p, p, p, None, None) == _lib.INVALID_ARG
    assert lib.fp4moe_mxfp4_as_nvfp4(ctypes.byref(nv), 2, 4, p, p, p, ctypes.c_void_p(0x10004), p, p,
                                     None) == _lib.MISALIGNED
    # NVFP4 TP shards: the logical width is whole 16-element scale blocks inside the kernel width
    assert lib.moe_route(ctypes.byref(_cfg(inter=768, inter_logical=700)), 8, *([p] * 13)) == _lib.UNSUPPORTED
    assert lib.moe_route(ctypes.byref(_cfg(inter=768, inter_logical=800)), 8, *([p] * 13)) == _lib.UNSUPPORTED
    assert lib.fp4moe_tensor_peak_probe(64, 10, p, None) == _lib.INVALID_ARG
    assert lib.fp4moe_tensor_peak_probe(128, 0, p, None) == _lib.INVALID_ARG
    assert lib.fp4moe_tensor_peak_probe(256, 10, None, None) == _lib.INVALID_ARG
