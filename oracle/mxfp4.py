"""MXFP4 expert weights and the TP3 virtual-padding shard plan.

Source: "Lucifer-CUTLASS TP3 virtual-padding audit".

* Section "TP3 shape plan". Routed MoE per-rank width is
  align_up(ceil(2048 / 3), 32) = 704, with a virtual global of 2112. The
  MXFP4 backend rounds the kernel-local width up to a multiple of 128, which
  gives 768 (section "Where the two sizes diverge").
* Sections "W13 happens to load correctly", "Packed W2 weight is wrong" and
  "W2 E8M0 scales are wrong". A shard is cut in LOGICAL elements and then
  converted to storage units: 1 per unpacked W13 row, 2 elements per packed
  W2 byte, 32 elements per E8M0 scale group. Every destination tail past the
  logical slice is zero.
* Section "2. CPU loader tests". The per-rank logical slices concatenate back
  to the source byte for byte.

MXFP4 follows OCP Microscaling v1.0. Each block of 32 elements along K shares
one E8M0 scale 2^X, with X = floor(log2(amax)) - 2, where 2 is the exponent of
the largest E2M1 power of two (4). X is clamped to [-127, 127], and an
all-zero block takes X = -127. Elements are E2M1_RNE_satfinite(v / 2^X), with
two per byte and the lower index in the low nibble.
"""
from __future__ import annotations

import math
from typing import NamedTuple

import numpy as np

from . import codecs

MX_BLOCK = 32
E2M1_EMAX = 2


def align_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


class TPPlan(NamedTuple):
    logical_per_rank: int   # 704 for 2048 / 3 aligned to 32
    virtual_global: int     # 2112
    kernel_local: int       # 768 after the backend's 128 rounding


def tp_plan(width: int, tp: int, align: int, kernel_align: int) -> TPPlan:
    local = align_up(math.ceil(width / tp), align)
    return TPPlan(local, local * tp, align_up(local, kernel_align))


def shard_units(width: int, plan: TPPlan, rank: int, unit: int):
    """(source offset, units copied, zero tail) of one rank, in storage units of ``unit`` elements."""
    start = rank * plan.logical_per_rank
    n = max(0, min(plan.logical_per_rank, width - start))
    assert start % unit == 0 and n % unit == 0 and plan.kernel_local % unit == 0
    return start // unit, n // unit, plan.kernel_local // unit - n // unit


def shard_axis(src: np.ndarray, axis: int, width: int, plan: TPPlan, rank: int, unit: int) -> np.ndarray:
    """Copy one rank's logical slice of ``src`` (axis in storage units) into a zeroed kernel-width buffer."""
    off, n, _ = shard_units(width, plan, rank, unit)
    shape = list(src.shape)
    shape[axis] = plan.kernel_local // unit
    dst = np.zeros(shape, dtype=src.dtype)
    sl_dst = [slice(None)] * src.ndim
    sl_src = [slice(None)] * src.ndim
    sl_dst[axis] = slice(0, n)
    sl_src[axis] = slice(off, off + n)
    dst[tuple(sl_dst)] = src[tuple(sl_src)]
    return dst


# ------------------------------------------------------------------ MXFP4 ----

def mx_quantize_rows(v: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """v [R, K] fp32 (K multiple of 32) -> (codes [R, K] 0..15, e8m0 scales [R, K/32])."""
    v = np.asarray(v, dtype=np.float32)
    R, K = v.shape
    blocks = v.reshape(R, K // MX_BLOCK, MX_BLOCK).astype(np.float64)
    amax = np.abs(blocks).max(axis=2)
    _, e = np.frexp(np.where(amax > 0, amax, 1.0))        # amax = m * 2^e, m in [0.5, 1)
    X = np.where(amax > 0, (e - 1) - E2M1_EMAX, -127)
    X = np.clip(X, -127, 127)
    scaled = blocks / np.ldexp(1.0, X)[:, :, None]         # exact (power of two)
    q = codecs.e2m1_encode(scaled.astype(np.float32)).reshape(R, K)
    return q, (X + 127).astype(np.uint8)


def mx_dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    R, K = q.shape
    el = codecs.e2m1_decode(q).reshape(R, K // MX_BLOCK, MX_BLOCK)
    return (el * codecs.e8m0_decode(s)[:, :, None]).reshape(R, K)
