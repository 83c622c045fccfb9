"""NVFP4 block quantisation and the 128x4 block-scale swizzle.

Quantisation follows the flow named on "Current Bug: CuTeDSLMoERunner" in
sections "Key Architecture: CuTeDSL NVFP4 MoE / Data Flow"
(quantize_activation_nvfp4 -> x_fp4, x_sf) and "Bug 5" / "Bug 6" (the
per-tensor activation global scale). The steps for a row v with
quant-direction global scale g, per 16-element block, are below. Every step
is IEEE fp32 with round-to-nearest-even.

  a   = max |v_i|                      (exact)
  s   = RN(RN(a / 6) * g)
  sf  = E4M3_RNE_satfinite(s)
  inv = 0 if sf == 0 else RN(g / decode(sf))
  q_i = E2M1_RNE_satfinite(RN(v_i * inv))

q_{2i} goes in the low nibble and q_{2i+1} in the high nibble of byte i. The
dequantised value is decode(q) * decode(sf) / g.

The global scale is g = RN(2688 / amax), where 2688 = 6 * 448 is the largest
|decoded element x decoded scale|. If amax = 0 then g = 1. Reading pinned by
"Current Bug", section "Bug 5". That section puts the checkpoint input_scale
at about 0.000286 for a calibration amax of about 0.77, and 0.77 / 2688 is
2.865e-4. It also says that too small a scale saturates the block scales at
448, which this convention reproduces.

Swizzle ("Blackwell 32_4_4 swizzle", "Current Bug" sections "Bug 1" and
"Bug 11"). For a scale matrix S[R, C], with R a multiple of 128 and C a
multiple of 4:

  byte(r, c) = ((r // 128) * (C // 4) + c // 4) * 512
               + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4

The pages name this layout but do not print it. This is the public 128x4
block-scale tile layout of the PTX ISA and cuBLAS for block-scaled MMA.
"""
from __future__ import annotations

import numpy as np

from . import codecs

F32 = np.float32
NVFP4_BLOCK = 16
GS_NUMERATOR = F32(6.0 * 448.0)   # 2688


def global_scale(amax) -> np.float32:
    """Quant-direction per-tensor global scale g = RN(2688 / amax); 1 when amax == 0."""
    a = F32(amax)
    if a == 0:
        return F32(1.0)
    return F32(GS_NUMERATOR / a)


def block_scales(v: np.ndarray, g) -> np.ndarray:
    """Step 2 of the quantiser before its E4M3 rounding: s = RN(RN(a / 6) * g) per 16-element block, fp32 [R, K/16].

    E4M3 rounding takes s above 448, the largest finite value, exactly when s > 464 (the midpoint to the next
    power-of-two step; the tie goes to 448, the even code): such a block's scale saturates.
    """
    v = np.asarray(v, dtype=F32)
    R, K = v.shape
    g = np.broadcast_to(np.asarray(g, dtype=F32).reshape(-1, 1) if np.ndim(g) else F32(g), (R, 1)).astype(F32)
    a = np.abs(v.reshape(R, K // NVFP4_BLOCK, NVFP4_BLOCK)).max(axis=2)
    return ((a / F32(6.0)).astype(F32) * g).astype(F32)


E4M3_SATURATES_ABOVE = 464.0


def quantize_rows(v: np.ndarray, g) -> tuple[np.ndarray, np.ndarray]:
    """NVFP4-quantise rows of fp32 values.

    v : [R, K] float32, with K a multiple of 16. g is an fp32 scalar or an [R]
    array of per-row global scales.
    Returns (codes [R, K] uint8 in 0..15, unpacked; scales [R, K/16] uint8 E4M3).
    """
    v = np.asarray(v, dtype=F32)
    R, K = v.shape
    assert K % NVFP4_BLOCK == 0
    g = np.broadcast_to(np.asarray(g, dtype=F32).reshape(-1, 1) if np.ndim(g) else F32(g), (R, 1)).astype(F32)
    blocks = v.reshape(R, K // NVFP4_BLOCK, NVFP4_BLOCK)
    s = block_scales(v, g)                                           # RN(RN(a/6) * g), a = max|v| exact
    sf = codecs.e4m3_encode(s)                                       # [R, K/16]
    sf_val = codecs.e4m3_decode(sf).astype(F32)                      # exact in fp32
    with np.errstate(divide="ignore"):
        inv = np.where(sf_val == 0, F32(0.0), (g / np.where(sf_val == 0, F32(1.0), sf_val)).astype(F32)).astype(F32)
    scaled = (blocks * inv[:, :, None]).astype(F32)                  # RN(v * inv)
    q = codecs.e2m1_encode(scaled).reshape(R, K)
    return q, sf


def pack_codes(q: np.ndarray) -> np.ndarray:
    """[R, K] codes 0..15 -> [R, K/2] bytes; element 2i in the low nibble."""
    q = np.asarray(q, dtype=np.uint8)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    out = np.empty((b.shape[0], b.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = b & 0xF
    out[:, 1::2] = b >> 4
    return out


def dequantize(q: np.ndarray, sf: np.ndarray, g) -> np.ndarray:
    """decode(q) * decode(sf) / g in fp64; q [R, K] codes, sf [R, K/16]."""
    R, K = q.shape
    g = np.asarray(g, dtype=np.float64).reshape(-1, 1) if np.ndim(g) else np.float64(g)
    el = codecs.E2M1_TABLE[np.asarray(q, dtype=np.uint8) & 0xF].reshape(R, K // NVFP4_BLOCK, NVFP4_BLOCK)
    sc = codecs.E4M3_TABLE[np.asarray(sf, dtype=np.uint8)][:, :, None]
    return (el * sc).reshape(R, K) / g


def swizzle_offset(r, c, C: int):
    """Byte offset of scale (r, c) in the 128x4-tiled layout of a matrix with C scale columns."""
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    return ((r // 128) * (C // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4


def swizzle(S: np.ndarray) -> np.ndarray:
    """S [R, C] (R multiple of 128, C multiple of 4) -> flat swizzled bytes (R*C)."""
    R, C = S.shape
    assert R % 128 == 0 and C % 4 == 0, (R, C)
    out = np.zeros(R * C, dtype=S.dtype)
    rr, cc = np.meshgrid(np.arange(R), np.arange(C), indexing="ij")
    out[swizzle_offset(rr, cc, C)] = S
    return out


def unswizzle(flat: np.ndarray, R: int, C: int) -> np.ndarray:
    rr, cc = np.meshgrid(np.arange(R), np.arange(C), indexing="ij")
    return np.asarray(flat)[swizzle_offset(rr, cc, C)]
