"""GPU: moe_forward_shared from two host threads at once.

The call forks the shared expert onto a side stream with events. Each host
thread gets its own side stream and event pair per device. Two threads, each
with its own layer buffers and workspace (the weights are shared) and its
own stream, run 20 forwards at the same time. Every output must equal, bit
for bit, the one computed by a single thread. A mix-up of events between the
threads would join a branch to the wrong call and break that.
"""
import threading

import numpy as np
import pytest

import synthgen as sg
from helpers import bits_to_torch, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _layers(wl, n):
    import torch
    from block_scaled_fp4_top_gb300 import api
    from synthgen import gpu as sgpu
    from helpers import make_layer
    base = make_layer(wl, wl.T)
    cfg = api.config(wl.H, wl.I, wl.E, wl.k, wl.T, wl.swiglu_limit, shared_inter=wl.shared_I)
    first = api.MoELayer(cfg)
    first.weights = base.weights
    first.router_w, first.router_bias = base.router_w, base.router_bias
    first.quantize_shared_weights(1, sgpu.shared_w1(wl))
    first.quantize_shared_weights(2, sgpu.shared_w2(wl))
    first.set_global_scales(0.5, 2.0)
    layers = [first]
    for _ in range(n - 1):
        other = api.MoELayer(cfg)
        other.weights, other.shared = first.weights, first.shared
        other.router_w, other.router_bias = first.router_w, first.router_bias
        other.set_global_scales(0.5, 2.0)
        layers.append(other)
    torch.cuda.synchronize()
    return layers


def test_two_threads_match_one_thread():
    import torch
    wl = sg.TINY_SHARED
    layers = _layers(wl, 2)
    reps = 20
    xs = [[bits_to_torch(sg.activations_bf16(wl, 500 + 100 * th + i)) for i in range(reps)] for th in range(2)]
    # reference: one thread, one stream, one layer
    ref = [[None] * reps for _ in range(2)]
    for th in range(2):
        for i in range(reps):
            y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device="cuda")
            layers[0].forward(xs[th][i], y)
            ref[th][i] = y
    torch.cuda.synchronize()
    assert layers[0].read_error() == 0

    got = [[torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device="cuda") for _ in range(reps)] for _ in range(2)]
    errors = []

    def run(th):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for i in range(reps):
                    layers[th].forward(xs[th][i], got[th][i], stream=s)
            s.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(th,)) for th in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for th in range(2):
        assert layers[th].read_error() == 0
        for i in range(reps):
            assert torch.equal(got[th][i].view(torch.int16), ref[th][i].view(torch.int16)), (th, i)
