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
* Section "Remaining kernel assumptions". The layer on a shard takes BF16
  activations with MXFP4 weights. Reading: h is rounded to bf16 before W2,
  because bf16 is the activation type of this variant. Each rank returns
  partial rows of the W2 output, and across ranks they sum to the
  full-width layer.

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
    """codes [R, K] and E8M0 scales [R, K/32] -> fp64 [R, K]."""
    R, K = q.shape
    el = codecs.E2M1_TABLE[np.asarray(q, dtype=np.uint8) & 0xF].reshape(R, K // MX_BLOCK, MX_BLOCK)
    return (el * codecs.E8M0_TABLE[np.asarray(s, dtype=np.uint8)][:, :, None]).reshape(R, K)


# ------------------------------------------------------- the MXFP4 layer ----

class MxExpert(NamedTuple):
    """One expert's kernel-local MXFP4 shard: codes unpacked, scales as E8M0 bytes.

    W13 rows [0, Ik) are the gate, [Ik, 2Ik) are up, each with its zero tail
    past the logical width. W2 is [H, Ik], whose columns past the logical
    width are zero codes with zero scale bytes.
    """
    w1_q: np.ndarray    # [2 Ik, H]
    w1_s: np.ndarray    # [2 Ik, H / 32]
    w2_q: np.ndarray    # [H, Ik]
    w2_s: np.ndarray    # [H, Ik / 32]


class MxCheckpoint(NamedTuple):
    """One expert's full-width MXFP4 tensors as a checkpoint stores them ("Packed W2 weight is wrong"):
    W13 codes unpacked one per row element, W2 codes packed two per byte, one E8M0 byte per 32 elements."""
    w13_q: np.ndarray       # [2 I, H] codes, gate rows first
    w13_s: np.ndarray       # [2 I, H / 32]
    w2_packed: np.ndarray   # [H, I / 2] bytes, element 2i in the low nibble
    w2_s: np.ndarray        # [H, I / 32]


def mx_checkpoint(w1_full: np.ndarray, w2_full: np.ndarray) -> MxCheckpoint:
    """Quantise one expert's full logical matrices: w1_full [2 I, H] (gate rows first), w2_full [H, I] fp32."""
    q1, s1 = mx_quantize_rows(w1_full)
    q2, s2 = mx_quantize_rows(w2_full)
    packed = (q2[:, 0::2] | (q2[:, 1::2] << 4)).astype(np.uint8)           # element 2i in the low nibble
    return MxCheckpoint(q1, s1, packed, s2)


def mx_shard_checkpoint(ck: MxCheckpoint, plan: TPPlan, rank: int) -> MxExpert:
    """Cut rank `rank`'s kernel-width shard out of a quantised checkpoint.

    The cut follows "Required loader changes": source offsets counted in
    logical elements and converted to each tensor's storage unit. W13 takes
    1 unpacked row per element. Packed W2 takes 2 elements per byte. W2
    scales take 32 elements per E8M0 group. The destination is zero-filled
    first.
    """
    I = ck.w13_q.shape[0] // 2
    gate_q = shard_axis(ck.w13_q[:I], 0, I, plan, rank, 1)
    up_q = shard_axis(ck.w13_q[I:], 0, I, plan, rank, 1)
    gate_s = shard_axis(ck.w13_s[:I], 0, I, plan, rank, 1)
    up_s = shard_axis(ck.w13_s[I:], 0, I, plan, rank, 1)
    packed_shard = shard_axis(ck.w2_packed, 1, I, plan, rank, 2)
    w2_q = np.empty((packed_shard.shape[0], packed_shard.shape[1] * 2), dtype=np.uint8)
    w2_q[:, 0::2] = packed_shard & 0xF
    w2_q[:, 1::2] = packed_shard >> 4
    w2_s = shard_axis(ck.w2_s, 1, I, plan, rank, 32)
    return MxExpert(np.concatenate([gate_q, up_q]), np.concatenate([gate_s, up_s]), w2_q, w2_s)


def mx_expert_shard(w1_full: np.ndarray, w2_full: np.ndarray, plan: TPPlan, rank: int) -> MxExpert:
    """Quantise one expert's full logical matrices to MXFP4, then cut rank `rank`'s shard.

    w1_full [2 I, H] (gate rows first), w2_full [H, I] fp32; I is the full width.
    """
    return mx_shard_checkpoint(mx_checkpoint(w1_full, w2_full), plan, rank)


# ------------------------------------- MXFP4 weights on the NVFP4 tensor-core form ----
#
# The block-scaled FP4 MMA that the NVFP4 layer runs multiplies an E2M1 code by an E4M3 scale per 16
# elements. An MX scale 2^X (E8M0, per 32) is a power of two, and E4M3 holds every power of two from 2^-9
# (the subnormal 0x01) to 2^8 (0x78). So with one power-of-two factor per matrix, G = X_max - 8, the MX
# value e2m1(q) * 2^X equals e2m1(q) * e4m3(sf) / gw exactly, for sf = E4M3(2^(X - G)) on both 16-element
# halves of the block and the quant-direction global scale gw = 2^-G. This holds for every block whose X
# lies in the 18-binade window [X_max - 17, X_max]; an all-zero block (E8M0 byte 0, zero codes) takes
# sf = 0. A nonzero block below the window has no exact form and is rejected.

E4M3_POW2_MIN = -9   # 0x01, the smallest subnormal
E4M3_POW2_MAX = 8    # 0x78 = 256; 512 is past the largest finite value, 448


def e4m3_pow2_byte(d: int) -> int:
    """The E4M3 byte of 2^d for -9 <= d <= 8 (bias 7: normals (d + 7) << 3 from d = -6; subnormals m / 8 * 2^-6)."""
    if not E4M3_POW2_MIN <= d <= E4M3_POW2_MAX:
        raise ValueError(f"2^{d} has no E4M3 form")
    return (d + 7) << 3 if d >= -6 else 1 << (d + 9)


def mx_as_nvfp4(q: np.ndarray, s: np.ndarray):
    """One matrix's MXFP4 weights (codes [R, K], E8M0 bytes [R, K/32]) as NVFP4 operands.

    Returns (codes [R, K] unchanged, E4M3 scale bytes [R, K/16], gw fp32) with
    nvfp4.dequantize(codes, sf, gw) == mx_dequantize(q, s) exactly.
    """
    s = np.asarray(s, dtype=np.uint8)
    if (s == 0xFF).any():
        raise ValueError("an E8M0 scale is NaN")
    live = s > 0
    if live.any() and (np.asarray(q, dtype=np.uint8).reshape(s.shape[0], s.shape[1], MX_BLOCK)[~live] & 0x7).any():
        raise ValueError("a block with E8M0 byte 0 has nonzero codes")
    X = s.astype(np.int64) - 127
    G = int(X[live].max()) - E4M3_POW2_MAX if live.any() else 0
    table = {d: e4m3_pow2_byte(d) for d in range(E4M3_POW2_MIN, E4M3_POW2_MAX + 1)}
    d = X - G
    if (live & (d < E4M3_POW2_MIN)).any():
        raise ValueError("a block lies more than 17 binades below the matrix's largest")
    sf32 = np.zeros(s.shape, dtype=np.uint8)
    sf32[live] = np.vectorize(table.__getitem__, otypes=[np.uint8])(d[live])
    sf = np.repeat(sf32, 2, axis=1)                                        # both 16-element halves
    return np.asarray(q, dtype=np.uint8), sf, np.float32(np.ldexp(1.0, -G))


def _bf16_round(v: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (round to nearest) -> bf16 (round to nearest even), returned as fp64."""
    b = np.ascontiguousarray(v.astype(np.float32)).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def mx_expert_out(qe: MxExpert, x: np.ndarray, limit: float) -> np.ndarray:
    """One expert's partial output rows for bf16-valued token rows x [n, H] (fp64), before the combine.

    [g; u] = W13~ x in fp64; h = silu(min(g, L)) * clamp(u, -L, L), rounded to
    bf16 (the W2 input of the bf16-activation variant); o = W2~ h.
    """
    from .moe import swiglu
    Ik = qe.w2_q.shape[1]
    W1 = mx_dequantize(qe.w1_q, qe.w1_s)                                   # [2 Ik, H]
    gu = x @ W1.T
    h = _bf16_round(swiglu(gu[:, :Ik], gu[:, Ik:], limit))
    return h @ mx_dequantize(qe.w2_q, qe.w2_s).T                            # [n, H]


def mx_moe_partials(x_bits: np.ndarray, ids: np.ndarray, expert, limit: float) -> np.ndarray:
    """Per-(token, j) partial rows o [n, k, H] (fp64) of the MXFP4 layer on one rank."""
    from .moe import bf16_to_f64
    x = bf16_to_f64(x_bits)
    n, k = ids.shape
    outs = np.zeros((n, k, x.shape[1]), dtype=np.float64)
    for e in np.unique(ids):
        tt, jj = np.nonzero(ids == e)
        outs[tt, jj] = mx_expert_out(expert(int(e)), x[tt], limit)
    return outs


def mx_moe_tokens(x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray, expert, limit: float) -> np.ndarray:
    """The MXFP4 layer on one rank: y = bf16(sum_j w_j o_j) in j order (``moe.combine``). Returns bf16 bits [n, H]."""
    from .moe import combine
    return combine(ids, w, mx_moe_partials(x_bits, ids, expert, limit))
