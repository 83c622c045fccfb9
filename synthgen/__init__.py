"""Seeded synthetic workloads for the block-scaled FP4 MoE layer.

This module is the one piece shared by the oracle (``oracle/``), the tests and
the benchmark. It draws numbers and describes workload shapes. It holds none
of the layer's arithmetic: no quantisation, routing, GEMM or combine.

Generator (counter-based, so any slice of any tensor can be drawn on its own):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014). The stream key of a tensor is
  ``mix64(seed * GOLDEN + tensor_id)``. Element ``i`` of the tensor is
  ``mix64(key + (i + 1) * GOLDEN)``. Everything is modulo 2**64.
* Approximate normal variate: Irwin-Hall sum of the four 16-bit fields of that
  64-bit word, ``S`` in ``[0, 262140]``, centred and scaled to unit variance:
  ``z = f32(S - 131070) * f32(sqrt(3) / 65536)``. Then ``value = f32(z * sigma)``.
  Each step is one IEEE fp32 operation with round-to-nearest-even.
  A second implementation (``synthgen/csrc/synth.cu``) therefore gives the same
  bits on the GPU.
* Bernoulli(p) mask: the high 32 bits of a second stream's word, compared with
  ``round(p * 2**32)``.
* bf16 rounding: round-to-nearest-even on the fp32 bit pattern.

The workload recipes (shapes, seeds and value distributions) follow the
DeepSeek-V4-Flash MoE shape named in "Lucifer-CUTLASS TP3 virtual-padding
audit", section "TP3 shape plan". That shape is hidden 4096, routed
intermediate 2048, 256 experts, top-k 6 and swiglu_limit 10.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
#: fp32 sqrt(3)/65536, bit pattern 0x37ddb3d7 (the GPU twin uses the same bits)
IH_SCALE = np.uint32(0x37DDB3D7).view(np.float32)
IH_CENTRE = 131070

# tensor ids (one independent stream per id)
TID_X = 1
TID_X_OUTLIER = 2
TID_ROUTER = 3
TID_W1 = 4
TID_W2 = 5
TID_ZIPF_PERM = 6
TID_SE_W1 = 7
TID_SE_W2 = 8


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = np.array([(seed * 0x9E3779B97F4A7C15 + tensor_id) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix64(z)[0]


def raw64(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Words ``start .. start+count-1`` of the stream (uint64)."""
    key = stream_key(seed, tensor_id)
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + i * GOLDEN)


def normal_f32(seed: int, tensor_id: int, start: int, count: int, sigma: float) -> np.ndarray:
    r = raw64(seed, tensor_id, start, count)
    m = np.uint64(0xFFFF)
    s = ((r & m) + ((r >> np.uint64(16)) & m) + ((r >> np.uint64(32)) & m) + (r >> np.uint64(48))).astype(np.int64)
    z = (s - IH_CENTRE).astype(np.float32) * IH_SCALE
    return (z * np.float32(sigma)).astype(np.float32)


def bernoulli_mask(seed: int, tensor_id: int, start: int, count: int, p: float) -> np.ndarray:
    thr = np.uint64(int(round(p * 2.0**32)))
    return (raw64(seed, tensor_id, start, count) >> np.uint64(32)) < thr


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 with round-to-nearest-even, returned as uint16 bit patterns."""
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# workload recipes
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int               # tokens per batch
    H: int               # hidden
    I: int               # routed intermediate (kernel-local)
    E: int               # experts
    k: int               # top-k
    swiglu_limit: float
    router_sigma: float  # std of router weights
    w_sigma: float       # std of expert weights before quantisation
    outlier_p: float     # Bernoulli probability of an activation outlier
    outlier_mult: float  # outlier multiplier
    model_seed: int      # seed of router and expert weights
    zipf_s: float = 0.0  # >0: router bias drawn from a Zipf popularity law
    zipf_beta: float = 0.0
    zipf_dead: int = 0   # experts at the tail of the Zipf ranking that get bias -1e4
    I_logical: int = 0   # logical intermediate (MXFP4 TP shard); 0 = same as I
    w_format: int = 0    # 0 = NVFP4, 1 = MXFP4, 2 = MXFP4 weights in the NVFP4 operand form (NVFP4 activations)
    shared_I: int = 0    # intermediate of the shared expert (block-FP8); 0 = none
    ep_first: int = 0    # expert parallelism: the layer holds experts [ep_first, ep_first + ep_count)
    ep_count: int = 0    # 0 = all experts

    @property
    def I_log(self) -> int:
        return self.I_logical or self.I


WARMUP_SEED = 1      # activation global-scale warmup batch
EVAL_SEED = 2        # batch compared against the oracle / timed
REPLAY_SEED0 = 1000  # graph replay i uses REPLAY_SEED0 + i

TINY = Workload("tiny", T=16, H=256, I=128, E=8, k=2, swiglu_limit=10.0,
                router_sigma=1.0 / 16.0, w_sigma=0.02, outlier_p=0.0, outlier_mult=1.0, model_seed=0)
DSV4_DECODE = Workload("dsv4_flash_decode_T64", T=64, H=4096, I=2048, E=256, k=6, swiglu_limit=10.0,
                       router_sigma=1.0 / 64.0, w_sigma=0.02, outlier_p=0.01, outlier_mult=20.0, model_seed=0)
DSV4_PREFILL_ZIPF = dataclasses.replace(DSV4_DECODE, name="dsv4_flash_prefill_zipf_T8192", T=8192,
                                        zipf_s=1.1, zipf_beta=1.0, zipf_dead=16)
TP3_MXFP4 = dataclasses.replace(DSV4_DECODE, name="dsv4_flash_tp3_rank0_mxfp4_T512", T=512, I=768,
                                I_logical=704, w_format=1, outlier_p=0.0, outlier_mult=1.0)
# the same shard's MXFP4 weights carried on the NVFP4 block-scaled path (fp4moe_mxfp4_as_nvfp4), with NVFP4
# activations
TP3_MXFP4_NVACT = dataclasses.replace(TP3_MXFP4, name="dsv4_flash_tp3_rank0_mxfp4w_nvfp4a_T512", w_format=2)
# the layer with DeepSeek-V4-Flash's shared expert (intermediate 2048, "TP3 shape plan")
TINY_SHARED = dataclasses.replace(TINY, name="tiny_shared", T=200, shared_I=256)
DSV4_DECODE_SHARED = dataclasses.replace(DSV4_DECODE, name="dsv4_flash_decode_shared_T64", shared_I=2048)
# one rank's share under expert parallelism: 48 of the 256 experts ("EP Configuration")
DSV4_DECODE_EP48 = dataclasses.replace(DSV4_DECODE, name="dsv4_flash_decode_ep48_T64", ep_first=96, ep_count=48)
GRAPH_SWEEP_T = tuple(2**i for i in range(13))  # 1 .. 4096

WORKLOADS = {w.name: w for w in (TINY, DSV4_DECODE, DSV4_PREFILL_ZIPF, TP3_MXFP4, TP3_MXFP4_NVACT, TINY_SHARED,
                                 DSV4_DECODE_SHARED,
                                 DSV4_DECODE_EP48)}


def activations_bf16(wl: Workload, seed: int, T: int | None = None, row0: int = 0) -> np.ndarray:
    """x [T, H] as bf16 bit patterns: N(0,1)-like, with Bernoulli outliers scaled by outlier_mult."""
    T = wl.T if T is None else T
    n = T * wl.H
    start = row0 * wl.H
    v = normal_f32(seed, TID_X, start, n, 1.0)
    if wl.outlier_p > 0.0:
        m = bernoulli_mask(seed, TID_X_OUTLIER, start, n, wl.outlier_p)
        v = np.where(m, v * np.float32(wl.outlier_mult), v).astype(np.float32)
    return f32_to_bf16_bits(v).reshape(T, wl.H)


def router_bf16(wl: Workload) -> np.ndarray:
    """Router weights [E, H] as bf16 bit patterns."""
    v = normal_f32(wl.model_seed, TID_ROUTER, 0, wl.E * wl.H, wl.router_sigma)
    return f32_to_bf16_bits(v).reshape(wl.E, wl.H)


def router_bias_f32(wl: Workload) -> np.ndarray | None:
    """Additive router logit bias [E] that makes expert popularity follow a Zipf law.

    b_e = beta * ln(p_e), where p_e is proportional to rank(e)^-s. Ranks come
    from a seeded permutation of the experts. The last ``zipf_dead`` ranks get
    b_e = -1e4, so those experts receive no tokens. Returns None for workloads
    without a bias.
    """
    if wl.zipf_s <= 0.0:
        return None
    keys = raw64(wl.model_seed, TID_ZIPF_PERM, 0, wl.E)
    order = np.argsort(keys, kind="stable")          # order[r] = expert with rank r+1
    rank = np.empty(wl.E, dtype=np.int64)
    rank[order] = np.arange(1, wl.E + 1)
    live = wl.E - wl.zipf_dead
    p = np.where(rank <= live, rank.astype(np.float64) ** (-wl.zipf_s), 0.0)
    p = p / p.sum()
    b = np.where(rank <= live, wl.zipf_beta * np.log(np.where(p > 0, p, 1.0)), -1.0e4)
    return b.astype(np.float32)


def expert_w1_f32(wl: Workload, e: int, I_full: int | None = None) -> np.ndarray:
    """W1 of expert e, [2*I_full, H] fp32: rows [0, I_full) gate, [I_full, 2*I_full) up."""
    I_full = wl.I_log if I_full is None else I_full
    n = 2 * I_full * wl.H
    return normal_f32(wl.model_seed, TID_W1, e * n, n, wl.w_sigma).reshape(2 * I_full, wl.H)


def expert_w2_f32(wl: Workload, e: int, I_full: int | None = None) -> np.ndarray:
    """W2 of expert e, [H, I_full] fp32 (output-major, K = intermediate contiguous)."""
    I_full = wl.I_log if I_full is None else I_full
    n = wl.H * I_full
    return normal_f32(wl.model_seed, TID_W2, e * n, n, wl.w_sigma).reshape(wl.H, I_full)


def shared_w1_f32(wl: Workload) -> np.ndarray:
    """W1 of the shared expert, [2*shared_I, H] fp32: rows [0, shared_I) gate, then up."""
    n = 2 * wl.shared_I * wl.H
    return normal_f32(wl.model_seed, TID_SE_W1, 0, n, wl.w_sigma).reshape(2 * wl.shared_I, wl.H)


def shared_w2_f32(wl: Workload) -> np.ndarray:
    """W2 of the shared expert, [H, shared_I] fp32."""
    n = wl.H * wl.shared_I
    return normal_f32(wl.model_seed, TID_SE_W2, 0, n, wl.w_sigma).reshape(wl.H, wl.shared_I)


def describe(wl: Workload) -> dict:
    d = dataclasses.asdict(wl)
    d["generator"] = "SplitMix64 counter streams, Irwin-Hall(4x16-bit) unit normal"
    return d


__all__ = [n for n in dir() if not n.startswith("_")] + ["_mix64"]
