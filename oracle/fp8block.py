"""Block-scaled FP8 (E4M3) codec and the shared expert, per token.

Test infrastructure: only the tests, the package's smoke check and the
benchmark's CPU baseline call this module. The product path never does.

What the pages fix:
* DeepSeek-V4-Flash has one shared expert with intermediate size 2048
  ("Lucifer-CUTLASS TP3 virtual-padding audit", "TP3 shape plan"). Under TP3
  each rank holds align_up(ceil(2048 / 3), 128) = 768 of its features; rank 2
  holds 512 real ones and 256 zeros ("Paths that already appear compatible").
* Its weights and their scales are block-FP8 (same section).
* It runs in the same captured step as the router and the routed MoE
  ("DSV4 -> vLLM: CUDA-Graph Safety / GPU-Native Requirements", Graph B:
  "Router + MoE + SE").

Readings where the pages stop:
* Block-FP8 is E4M3 with one fp32 scale per block: 128 x 128 blocks for
  weights and 1 x 128 groups along K for activations. This is the recipe of
  the DeepSeek-V3 technical report (section 3.3, "FP8 training"). The 128
  alignment of the shared shard keeps the blocks whole.
* A block's scale is s = RN_f32(amax / 448). Its codes are
  E4M3_RNE_satfinite(RN_f32(v / s)). A block with s == 0 (all zero, or an
  amax too small for s to be a nonzero fp32) has code 0 everywhere.
  Dequantisation is q * s.
* The shared expert has the routed experts' FFN form: W1 rows [0, Is) are the
  gate and rows [Is, 2Is) are up; h is the clamped SwiGLU with the layer's
  limit. h is rounded to fp32 and quantised per 1 x 128 group, like x.
* Its output enters the combine's sum with weight 1, after the routed terms:
  y_t = bf16(sum_j w_t,j * o_j + o_shared,t).
"""
from __future__ import annotations

import math
from typing import NamedTuple

import numpy as np

from . import codecs
from .moe import bf16_to_f64, swiglu

F32 = np.float32
BLOCK = 128
E4M3_MAX = F32(448.0)


def block_scale(amax) -> np.float32:
    """s = RN_f32(amax / 448) for one block's fp32 amax."""
    return F32(F32(amax) / E4M3_MAX)


def encode_block(v: np.ndarray, s) -> np.ndarray:
    """E4M3 codes of the fp32 values v under scale s; all zero when s == 0."""
    v = np.asarray(v, dtype=F32)
    if F32(s) == 0:
        return np.zeros(v.shape, dtype=np.uint8)
    with np.errstate(over="ignore"):
        r = (v / F32(s)).astype(F32)
    return codecs.e4m3_encode(r)


def quantize_groups(v: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Activations [n, K] fp32 -> codes [n, K] u8 and scales [n, K/128] fp32 (1 x 128 groups)."""
    v = np.asarray(v, dtype=F32)
    n, K = v.shape
    assert K % BLOCK == 0
    q = np.zeros((n, K), dtype=np.uint8)
    s = np.zeros((n, K // BLOCK), dtype=F32)
    for t in range(n):
        for g in range(K // BLOCK):
            blk = v[t, g * BLOCK:(g + 1) * BLOCK]
            s[t, g] = block_scale(np.abs(blk).max())
            q[t, g * BLOCK:(g + 1) * BLOCK] = encode_block(blk, s[t, g])
    return q, s


def quantize_blocks(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Weights [R, K] fp32 -> codes [R, K] u8 and scales [R/128, K/128] fp32 (128 x 128 blocks)."""
    w = np.asarray(w, dtype=F32)
    R, K = w.shape
    assert R % BLOCK == 0 and K % BLOCK == 0
    q = np.zeros((R, K), dtype=np.uint8)
    s = np.zeros((R // BLOCK, K // BLOCK), dtype=F32)
    for i in range(R // BLOCK):
        for j in range(K // BLOCK):
            blk = w[i * BLOCK:(i + 1) * BLOCK, j * BLOCK:(j + 1) * BLOCK]
            s[i, j] = block_scale(np.abs(blk).max())
            q[i * BLOCK:(i + 1) * BLOCK, j * BLOCK:(j + 1) * BLOCK] = encode_block(blk, s[i, j])
    return q, s


def dequantize_groups(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    return codecs.e4m3_decode(q) * np.repeat(s.astype(np.float64), BLOCK, axis=1)


def dequantize_blocks(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    full = np.repeat(np.repeat(s.astype(np.float64), BLOCK, axis=0), BLOCK, axis=1)
    return codecs.e4m3_decode(q) * full


class SharedExpert(NamedTuple):
    """The shared expert's block-FP8 weights in logical order."""
    w1_q: np.ndarray   # [2Is, H] codes, rows [0, Is) gate, [Is, 2Is) up
    w1_s: np.ndarray   # [2Is/128, H/128]
    w2_q: np.ndarray   # [H, Is]
    w2_s: np.ndarray   # [H/128, Is/128]


def quantize_shared(w1: np.ndarray, w2: np.ndarray) -> SharedExpert:
    q1, s1 = quantize_blocks(w1)
    q2, s2 = quantize_blocks(w2)
    return SharedExpert(q1, s1, q2, s2)


def shared_out(x_bits: np.ndarray, se: SharedExpert, limit: float, quantize_activations: bool = True) -> np.ndarray:
    """o_shared [n, H] fp64 for bf16 token rows x_bits [n, H].

    quantize_activations=False replaces both activation codecs by the identity.
    """
    x = bf16_to_f64(x_bits)
    Is = se.w2_q.shape[1]
    xt = dequantize_groups(*quantize_groups(x.astype(F32))) if quantize_activations else x
    gu = xt @ dequantize_blocks(se.w1_q, se.w1_s).T
    h = swiglu(gu[:, :Is], gu[:, Is:], limit)
    ht = dequantize_groups(*quantize_groups(h.astype(F32))) if quantize_activations else h
    return ht @ dequantize_blocks(se.w2_q, se.w2_s).T


def tp_shard(w1: np.ndarray, w2: np.ndarray, rank: int, world: int) -> tuple[np.ndarray, np.ndarray]:
    """One rank's fp32 shard of the shared expert under TP along the intermediate axis.

    Each rank holds align_up(ceil(I / world), 128) features, zero past the end
    of the tensor ("TP3 shape plan": 2048 over 3 ranks gives 768, 768 and 512
    real features).
    """
    I = w2.shape[1]
    per = math.ceil(math.ceil(I / world) / BLOCK) * BLOCK
    a, n = rank * per, max(0, min(per, I - rank * per))
    s1 = np.zeros((2 * per, w1.shape[1]), dtype=F32)
    s1[:n] = w1[a:a + n]
    s1[per:per + n] = w1[I + a:I + a + n]
    s2 = np.zeros((w2.shape[0], per), dtype=F32)
    s2[:, :n] = w2[:, a:a + n]
    return s1, s2
