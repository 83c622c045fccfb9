"""GPU: the CUDA-graph batch sweep at the DeepSeek-V4-Flash decode shape.

One graph is captured per token bucket T in {1, 2, 4, ..., 4096} over buffers
of fixed capacity, and replayed 100 times. Before every replay the input
buffer is refilled, outside the graph, with a freshly seeded batch (seed
1000 + replay) drawn on the GPU by the generator's bit-identical twin.

Every replay must:
* equal the eager call on the same input, bit for bit;
* leave the device error word at zero.
Replays 0 and 99 of every bucket also compare their top-k ids for all tokens
with the oracle's routing. A few sampled tokens of those replays also compare
their output rows with the oracle's layer, within the float bar.

The captured step must contain no host synchronisation, allocation or
device-value branch ("CUDA-Graph Safety / GPU-Native Requirements",
SECTION B). Capture itself would fail on any of them, and the replay/eager
equality shows the graph reads its inputs fresh each time.
"""
import numpy as np
import pytest

import synthgen as sg
from helpers import OracleExperts, bits_to_torch, ensure_built, float_parity, make_layer, torch_to_bits
from oracle import moe

pytestmark = pytest.mark.gpu

REPLAYS = 100
CHECKED = (0, REPLAYS - 1)
ORACLE_TOKENS = {1: [0], 64: [37], 4096: [4095]}  # bucket -> token rows checked against the oracle layer


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_graph_sweep_replays():
    import torch
    from synthgen import gpu as sgpu
    wl = sg.DSV4_DECODE
    Tmax = max(sg.GRAPH_SWEEP_T)
    layer = make_layer(wl, Tmax)
    layer.calibrate(bits_to_torch(sg.activations_bf16(wl, sg.WARMUP_SEED, T=wl.T)))
    gs1, gs2 = np.float32(layer.gs1.item()), np.float32(layer.gs2.item())
    wr = sg.router_bf16(wl)
    experts = OracleExperts(wl)
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
                rows = ORACLE_TOKENS.get(T, [])
                if rows:
                    y_ref = moe.moe_tokens(x_bits[rows], ids_ref[rows], w_ref[rows], experts, gs1, gs2,
                                           wl.swiglu_limit)
                    y_got = torch_to_bits(y)[rows]
                    float_parity(sg.bf16_bits_to_f32(y_got), sg.bf16_bits_to_f32(y_ref))
        torch.cuda.synchronize()
        assert layer.read_error() == 0
        del g
