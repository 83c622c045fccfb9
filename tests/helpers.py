"""Shared test utilities: bf16 conversions, GPU layer set-up from the seeded
generator, a lazily filled oracle expert table, and the float parity check."""
from __future__ import annotations

import os

import numpy as np

import synthgen as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def ensure_built():
    from block_scaled_fp4_top_gb300 import build as libbuild
    from synthgen import build as synthbuild
    libbuild.build()
    synthbuild.build()


def bits_to_torch(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def torch_to_bits(t) -> np.ndarray:
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# Bytes [64, 80) of the workspace header: the two grouped GEMMs' schedule counter pairs (chunks or pool tiles
# taken, CTAs done). The library keeps them at zero between calls, so that no call needs a memset.
SCHED_COUNTERS = slice(64, 80)


def assert_sched_counters_zero(ws):
    """The grouped GEMMs' schedule counters are back at zero (after a synchronize)."""
    words = ws[SCHED_COUNTERS].cpu().numpy().view(np.int32)
    assert (words == 0).all(), f"schedule counters left at {words.tolist()}"


def make_layer(wl: sg.Workload, max_tokens: int, chunk: int = 16):
    """GPU layer whose weights come from the GPU twin of the generator, quantised by the library."""
    import torch
    from block_scaled_fp4_top_gb300 import api
    from synthgen import gpu as sgpu
    cfg = api.config(wl.H, wl.I, wl.E, wl.k, max_tokens, wl.swiglu_limit)
    layer = api.MoELayer(cfg)
    for e0 in range(0, wl.E, chunk):
        n = min(chunk, wl.E - e0)
        w1 = sgpu.expert_w1(wl, e0, n)
        layer.quantize_weights(1, e0, w1)
        del w1
        w2 = sgpu.expert_w2(wl, e0, n)
        layer.quantize_weights(2, e0, w2)
        del w2
    bias = sg.router_bias_f32(wl)
    layer.set_router(sgpu.router(wl), None if bias is None else torch.from_numpy(bias).cuda())
    torch.cuda.synchronize()
    return layer


class OracleExperts:
    """Expert weights for the oracle: numpy generator + oracle quantiser, cached per expert."""

    def __init__(self, wl: sg.Workload):
        self.wl = wl
        self.cache = {}

    def __call__(self, e: int):
        from oracle import moe
        if e not in self.cache:
            self.cache[e] = moe.quantize_expert(sg.expert_w1_f32(self.wl, e), sg.expert_w2_f32(self.wl, e))
        return self.cache[e]


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """One unit in the last place of bf16 at |v| (8 significant bits; subnormals: 2^-133)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a >= 2.0 ** -126, a, 1.0)))
    return np.where(a >= 2.0 ** -126, 2.0 ** (e - 7), 2.0 ** -133)


def float_parity(got: np.ndarray, ref: np.ndarray, rel_l2: float = 1e-2, max_abs_rms: float = 2e-2,
                 bf16: bool = False, bf16_terms=None):
    """The layer's float bar: relative L2 <= 1e-2 and max |err| <= 2e-2 * RMS(ref).

    bf16=True: got and ref are both bf16 outputs, each rounded once from its own fp32 (GPU) or fp64 (oracle)
    sum. Where 2e-2 * RMS is finer than one bf16 ulp of an element, a sum that lands on the other side of a
    rounding boundary moves that element by one ulp whichever side is right, so an element's bar is
    max(2e-2 * RMS, ulp(ref)).
    bf16_terms=[t0, t1, ...]: got is a sum of bf16-rounded parts (tensor- or expert-parallel ranks) and ref
    the bf16 whole. Each rounding adds up to half an ulp of its own value, so an element's bar is
    2e-2 * RMS + (sum of ulp(t_i) + ulp(ref)) / 2.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), "non-finite output"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    rms = np.sqrt(np.mean(ref ** 2))
    bar = np.full(ref.shape, max_abs_rms * rms)
    if bf16:
        bar = np.maximum(bar, bf16_ulp(ref))
    if bf16_terms is not None:
        bar = bar + 0.5 * (sum(bf16_ulp(t) for t in bf16_terms) + bf16_ulp(ref))
    err = np.abs(got - ref)
    mx = err.max() if got.size else 0.0
    over = int((err > bar).sum())
    assert rel <= rel_l2 and over == 0, (f"rel L2 {rel:.3e} (<= {rel_l2}), max abs {mx:.3e} (bar {max_abs_rms} * rms "
                                         f"{rms:.3e}{' or the rounding slack' if bf16 or bf16_terms else ''}), "
                                         f"{over} elements over their bar")
    return rel, mx / rms if rms > 0 else 0.0


def tile_weights(packed: np.ndarray, rows_per_expert: int) -> np.ndarray:
    """Row-major packed codes [E*R][K/2] -> the pre-tiled weight layout of include/fp4moe.h.

    16 KB blocks [expert][row tile][k stage]; row i of a block holds 128 bytes
    whose 16-byte chunk j sits at i*128 + (j ^ (i % 8))*16; K is zero-padded to 256.
    """
    n_rows, kbytes = packed.shape
    E = n_rows // rows_per_expert
    kst = (kbytes + 127) // 128
    padded = np.zeros((n_rows, kst * 128), dtype=np.uint8)
    padded[:, :kbytes] = packed
    # [E, row_tiles, 128 rows, k_stages, 8 chunks, 16 bytes]
    t = padded.reshape(E, rows_per_expert // 128, 128, kst, 8, 16)
    i = np.arange(128)[:, None]
    j = np.arange(8)[None, :]
    out = np.zeros_like(t)
    out[:, :, i, :, j ^ (i % 8), :] = t[:, :, i, :, j, :]
    return out.transpose(0, 1, 3, 2, 4, 5).reshape(-1)


def untile_weights(flat: np.ndarray, n_rows: int, kbytes: int, rows_per_expert: int) -> np.ndarray:
    E = n_rows // rows_per_expert
    kst = (kbytes + 127) // 128
    t = flat.reshape(E, rows_per_expert // 128, kst, 128, 8, 16).transpose(0, 1, 3, 2, 4, 5)
    i = np.arange(128)[:, None]
    j = np.arange(8)[None, :]
    out = np.zeros_like(t)
    out[:, :, i, :, j, :] = t[:, :, i, :, j ^ (i % 8), :]
    return out.reshape(n_rows, kst * 128)[:, :kbytes]


def dump(name: str, **arrays):
    """Save arrays for offline diagnosis when FP4MOE_DUMP_DIR is set."""
    d = os.environ.get("FP4MOE_DUMP_DIR")
    if d:
        os.makedirs(d, exist_ok=True)
        np.savez_compressed(os.path.join(d, name + ".npz"), **arrays)
