"""GPU: moe_route_noalloc, the workspace-free routing call, against moe_route.

moe_route_noalloc keeps its histograms, router-row norms and partial router
tiles in one scratch array owned by the library instead of a caller
workspace. Its outputs must
match those of moe_route on the same inputs. Here that holds for two calls in
a row, and again after a call of the other layout path (a small T and a large
T), because the second call finds the scratch as the first call left it. The
file runs last so that it also passes after every other test has used the
library; it builds what it needs itself, so it passes alone too.
"""
import numpy as np
import pytest

import synthgen as sg
from helpers import bits_to_torch, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _outputs(wl, T, cap):
    import torch
    i32 = dict(dtype=torch.int32, device="cuda")
    n = max(T, 1)
    return dict(logits=torch.full((n, wl.E), -3.0, dtype=torch.float32, device="cuda"),
                ids=torch.full((n * wl.k,), -5, **i32),
                w=torch.full((n * wl.k,), -1.0, dtype=torch.float32, device="cuda"),
                counts=torch.full((wl.E,), -9, **i32), offsets=torch.full((wl.E,), -9, **i32),
                poff=torch.full((wl.E,), -9, **i32), slot=torch.full((n * wl.k,), -9, **i32),
                por=torch.full((cap,), -7, **i32))


def _inputs(wl, T, seed):
    import torch
    if T > 0:
        x = bits_to_torch(sg.activations_bf16(wl, seed, T=T))
    else:  # an empty tensor has no storage; the call wants a valid pointer it never reads
        x = torch.zeros(1, wl.H, dtype=torch.bfloat16, device="cuda")
    wr = bits_to_torch(sg.router_bf16(wl))
    bias = sg.router_bias_f32(wl)
    return x, wr, (None if bias is None else torch.from_numpy(bias).cuda())


def _route_both(wl, T, seed, calls=2, null_err=False):
    """moe_route once, then `calls` back-to-back moe_route_noalloc calls on the same inputs (with err NULL when
    null_err: errors then go to the scratch's own word, which each call clears)."""
    import torch
    from block_scaled_fp4_top_gb300 import api
    cfg = api.config(wl.H, wl.I, wl.E, wl.k, max(T, 1), wl.swiglu_limit)
    cap = api.capacity_rows(cfg, T)
    x, wr, bias = _inputs(wl, T, seed)
    ref = _outputs(wl, T, cap)
    ws = torch.zeros(api.workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    api.moe_route(cfg, T, x, wr, bias, ref["logits"], ref["ids"], ref["w"], ref["counts"], ref["offsets"],
                  ref["poff"], ref["slot"], ref["por"], ws)
    torch.cuda.synchronize()
    assert api.fp4moe_read_error(ws) == 0
    runs = []
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(calls):
        got = _outputs(wl, T, cap)
        api.moe_route_noalloc(cfg, T, x, wr, bias, got["logits"], got["ids"], got["w"], got["counts"],
                              got["offsets"], got["poff"], got["slot"], got["por"], None if null_err else err)
        runs.append(got)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    return ref, [{k: v.cpu().numpy() for k, v in g.items()} for g in runs]


def _compare(ref, got, T, k):
    R = int(ref["poff"][-1])
    n = T * k
    for key in ("counts", "offsets", "poff"):
        assert (got[key] == ref[key]).all(), key
    assert (got["ids"][:n] == ref["ids"][:n]).all()
    assert (got["slot"][:n] == ref["slot"][:n]).all()
    assert (got["por"][:R] == ref["por"][:R]).all()
    # floating outputs: the same kernels on the same inputs, so the tolerance is tight
    np.testing.assert_allclose(got["logits"][:T], ref["logits"][:T], rtol=1e-6, atol=0)
    np.testing.assert_allclose(got["w"][:n], ref["w"][:n], rtol=1e-6, atol=0)


@pytest.mark.parametrize("wl,T", [(sg.DSV4_DECODE, 64), (sg.DSV4_PREFILL_ZIPF, 8192), (sg.DSV4_DECODE, 64)])
def test_noalloc_matches_moe_route_two_calls_in_a_row(wl, T):
    ref, runs = _route_both(wl, T, sg.EVAL_SEED, calls=2)
    for got in runs:
        _compare(ref, got, T, wl.k)


def test_noalloc_with_no_error_word():
    ref, runs = _route_both(sg.DSV4_DECODE, 64, sg.EVAL_SEED, calls=2, null_err=True)
    for got in runs:
        _compare(ref, got, 64, sg.DSV4_DECODE.k)


def test_noalloc_takes_no_device_memory_eager_or_captured():
    """After a first eager call, further calls (eager, and captured in a CUDA graph and replayed) leave the
    device's free memory as it was: the call allocates nothing. The replay gives the eager outputs."""
    import torch
    from block_scaled_fp4_top_gb300 import api
    wl, T = sg.DSV4_DECODE, 64
    cfg = api.config(wl.H, wl.I, wl.E, wl.k, T, wl.swiglu_limit)
    cap = api.capacity_rows(cfg, T)
    x, wr, bias = _inputs(wl, T, sg.EVAL_SEED)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    eager, cap_out = _outputs(wl, T, cap), _outputs(wl, T, cap)
    call = lambda o, stream=None: api.moe_route_noalloc(cfg, T, x, wr, bias, o["logits"], o["ids"], o["w"],
                                                        o["counts"], o["offsets"], o["poff"], o["slot"], o["por"],
                                                        err, stream)
    call(eager)                                             # the first call on the device, outside capture
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    call(eager)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call(cap_out, s)
    torch.cuda.current_stream().wait_stream(s)
    free1 = torch.cuda.mem_get_info()[0]                    # the graph itself may hold memory; the call adds none
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free1
    assert int(err.item()) == 0
    for key in eager:
        assert torch.equal(eager[key], cap_out[key]), key


def test_noalloc_tiny_and_empty():
    for T in (16, 5, 0):
        ref, runs = _route_both(sg.TINY, T, sg.EVAL_SEED, calls=2)
        if T == 0:
            for got in runs:
                assert (got["counts"] == 0).all() and (got["poff"] == 0).all()
            continue
        for got in runs:
            _compare(ref, got, T, sg.TINY.k)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import ctypes
    import torch
    from block_scaled_fp4_top_gb300 import _lib, api
    lib = _lib.load()
    p = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails validation first
    args = [p] * 11 + [None, None]
    big = api.config(4096, 2048, 256, 6, 16384, 10.0)
    assert lib.moe_route_noalloc(ctypes.byref(big), 8193, *args) == _lib.CAPACITY
    many = api.config(4096, 2048, 512, 6, 64, 10.0)
    assert lib.moe_route_noalloc(ctypes.byref(many), 8, *args) == _lib.CAPACITY
    dec = api.config(4096, 2048, 256, 6, 64, 10.0)
    no_logits = [p] * 3 + [None] + [p] * 7 + [None, None]
    assert lib.moe_route_noalloc(ctypes.byref(dec), 8, *no_logits) == _lib.INVALID_ARG
    with pytest.raises(api.Fp4MoeError, match="FP4MOE_CAPACITY"):
        x = torch.zeros(1, 4096, dtype=torch.bfloat16, device="cuda")
        api.moe_route_noalloc(big, 8193, x, x, None, x, x, x, x, x, x, x, x)
