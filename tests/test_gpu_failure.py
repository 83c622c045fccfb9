"""GPU: failure detection through the bounded waits, with no GPU fault.

Every spin-wait in the kernels gives up after a time limit, sets
FP4MOE_ERR_TIMEOUT in the error word and lets its kernel return.
fp4moe_selftest_wait_timeout drives that same routine into its limit: it waits
on an mbarrier that nothing arrives at. These tests check three things.
* The host sees the error bit and the context stays usable.
* A forward pass whose error word already holds the abort bit skips its GEMMs
  and finishes promptly instead of waiting.
* After the word is cleared, the layer computes the same output as before.
Nothing here traps, faults or hangs a GPU.
"""
import time

import numpy as np
import pytest

import synthgen as sg
from helpers import assert_sched_counters_zero, bits_to_torch, ensure_built, make_layer, torch_to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_wait_runs_out_and_reports():
    import torch
    from block_scaled_fp4_top_gb300 import _lib, api
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    res = torch.full((4,), 7, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    api.fp4moe_selftest_wait_timeout(err, 5_000_000, res)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(res[0].item()) == 0, "the wait completed although nothing arrived"
    assert int(err[0].item()) & _lib.ERR_TIMEOUT
    assert 0.004 <= dt < 2.0
    # the context is still usable: a plain copy round-trips
    a = torch.arange(1000, device="cuda")
    assert int(a.sum().item()) == 499500


def test_limit_is_range_checked():
    import torch
    from block_scaled_fp4_top_gb300 import api
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    for bad in (0, 999_999, 50_000_001):
        with pytest.raises(api.Fp4MoeError, match="INVALID_ARG"):
            api.fp4moe_selftest_wait_timeout(err, bad, res)


def test_abort_bit_poisons_then_recovers():
    import torch
    from block_scaled_fp4_top_gb300 import _lib, api
    wl = sg.TINY
    layer = make_layer(wl, wl.T)
    layer.calibrate(bits_to_torch(sg.activations_bf16(wl, sg.WARMUP_SEED)))
    x = bits_to_torch(sg.activations_bf16(wl, sg.EVAL_SEED))
    y_ref = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device="cuda")
    layer.forward(x, y_ref)
    torch.cuda.synchronize()
    assert layer.read_error() == 0
    ref = torch_to_bits(y_ref)

    # a timeout lands in the layer's own error word (the first 4 bytes of its workspace)
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    api.fp4moe_selftest_wait_timeout(layer.ws, 2_000_000, res)
    y = torch.empty_like(y_ref)
    t0 = time.perf_counter()
    layer.forward(x, y)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 2.0, "a poisoned call must not wait out its limits"
    assert layer.read_error(clear=True) & _lib.ERR_TIMEOUT
    assert_sched_counters_zero(layer.ws)   # the skipped GEMMs still leave their schedule counters at zero

    layer.forward(x, y)
    torch.cuda.synchronize()
    assert layer.read_error() == 0
    assert np.array_equal(torch_to_bits(y), ref)
