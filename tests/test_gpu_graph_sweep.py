"""GPU: the CUDA-graph batch sweep at the DeepSeek-V4-Flash decode shape.

One graph is captured per token bucket T in {1, 2, 4, ..., 4096} over buffers
of fixed capacity, and replayed 100 times. Before every replay the input
buffer is refilled, outside the graph, with a freshly seeded batch (seed
1000 + replay) drawn on the GPU by the generator's bit-identical twin.

Every replay must:
* equal the eager call on the same input, bit for bit;
* leave the device error word at zero.
Replays 0 and 99 of every bucket also compare their top-k ids and weights for
all tokens with the oracle's routing, and output rows with the oracle's layer
(with the oracle's own warm-up scales) within the float bar: every token of
the buckets T <= 64; the first, the last and two seeded tokens of every
larger bucket.

The captured step must contain no host synchronisation, allocation or
device-value branch ("CUDA-Graph Safety / GPU-Native Requirements",
SECTION B). Capture itself would fail on any of them, and the replay/eager
equality shows the graph reads its inputs fresh each time.
"""
import numpy as np
import pytest

import synthgen as sg
from helpers import assert_sched_counters_zero, bits_to_torch, ensure_built, float_parity, make_layer, torch_to_bits
from oracle import moe

pytestmark = pytest.mark.gpu

REPLAYS = 100
CHECKED = (0, REPLAYS - 1)


def oracle_tokens(T: int, replay: int) -> np.ndarray:
    """Token rows whose outputs are checked against the oracle: all of them up to T = 64, else the first, the
    last and two seeded others."""
    if T <= 64:
        return np.arange(T)
    rng = np.random.default_rng(1000 * T + replay)
    return np.sort(np.concatenate([[0, T - 1], rng.choice(np.arange(1, T - 1), 2, replace=False)]))


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_graph_sweep_replays(oracle_svc):
    import torch
    from synthgen import gpu as sgpu
    wl = sg.DSV4_DECODE
    Tmax = max(sg.GRAPH_SWEEP_T)
    layer = make_layer(wl, Tmax)
    xw = sg.activations_bf16(wl, sg.WARMUP_SEED, T=wl.T)
    layer.calibrate(bits_to_torch(xw))
    gs1, gs2 = oracle_svc.calibrate(wl, xw)
    assert float(layer.gs1.item()) == float(gs1)
    assert float(layer.gs2.item()) == pytest.approx(float(gs2), rel=1e-5)
    wr = sg.router_bf16(wl)
    checked_x, checked_y, labels = [], [], []   # rows compared with the oracle's layer after the sweep
    dev = "cuda"
    for T in sg.GRAPH_SWEEP_T:
        x = torch.empty(T, wl.H, dtype=torch.bfloat16, device=dev)
        y = torch.empty(T, wl.H, dtype=torch.bfloat16, device=dev)
        ids = torch.empty(T * wl.k, dtype=torch.int32, device=dev)
        w = torch.empty(T * wl.k, dtype=torch.float32, device=dev)
        y_e = torch.empty_like(y)
        ids_e = torch.empty_like(ids)
        sgpu.activations(wl, sg.REPLAY_SEED0, T=T, out=x)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            layer.forward(x, y, ids, w)  # first call outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer.forward(x, y, ids, w)
        for i in range(REPLAYS):
            sgpu.activations(wl, sg.REPLAY_SEED0 + i, T=T, out=x)
            g.replay()
            layer.forward(x, y_e, ids_e, None)
            assert torch.equal(y, y_e) and torch.equal(ids, ids_e), f"T={T} replay {i}: graph and eager differ"
            if i in CHECKED:
                torch.cuda.synchronize()
                assert layer.read_error() == 0
                x_bits = sg.activations_bf16(wl, sg.REPLAY_SEED0 + i, T=T)
                ids_ref, w_ref = moe.topk_softmax(moe.router_logits(x_bits, wr, None), wl.k)
                got_ids = ids.cpu().numpy().reshape(T, wl.k)
                assert (got_ids == ids_ref).all(), f"T={T} replay {i}: top-k ids differ from the oracle"
                assert np.allclose(w.cpu().numpy().reshape(T, wl.k), w_ref, rtol=3e-6, atol=1e-7)
                rows = oracle_tokens(T, i)
                checked_x.append(x_bits[rows])
                checked_y.append(torch_to_bits(y)[rows])
                labels.append((T, i))
        torch.cuda.synchronize()
        assert layer.read_error() == 0
        assert_sched_counters_zero(layer.ws)   # the replays leave the GEMMs' counters as they found them
        del g
    # every checked row of every bucket against the oracle, in one pass over the experts
    ref = oracle_svc.layer(wl, checked_x, gs1, gs2)
    assert sum(len(r) for r in checked_x) == 2 * (127 + 4 * 6)
    for (T, i), got, (y_ref, _, _) in zip(labels, checked_y, ref):
        try:
            float_parity(sg.bf16_bits_to_f32(got), sg.bf16_bits_to_f32(y_ref), bf16=True)
        except AssertionError as exc:
            raise AssertionError(f"T={T} replay {i}: {exc}") from None
