"""Router, softmax top-k, clamped SwiGLU and the per-token routed-MoE layer.

The data flow is the one on "Current Bug: CuTeDSLMoERunner", section
"Key Architecture: CuTeDSL NVFP4 MoE / Data Flow":

  x (bf16) -> route -> L1 NVFP4 quantise -> grouped GEMM W13 (gate | up)
    -> SiLU(gate) * up -> L2 NVFP4 quantise -> grouped GEMM W2
    -> weighted scatter_add -> y (bf16)

The oracle states this per token. It does not scatter, pad or tile:

  l_t   = RN_f32( sum_h x[t,h] * Wr[e,h] )  (fp64 sum rounded once to fp32), plus an optional fp32 bias
  S_t   = the top-k experts of l_t, ordered by descending logit, ties to the lower expert id
  w_t,j = exp(l_j - l_max) / sum_{i in S_t} exp(l_i - l_max)  (softmax over the selected logits)
  x~_t  = dequant(quant(x_t, gs1))
  for each e in S_t (fp64):
      [g; u] = alpha-scaled W1~_e x~_t
      h      = silu(min(g, L)) * clamp(u, -L, L)
      h~     = dequant(quant(RN_f32(h), gs2))
      o_e    = W2~_e h~, returned in bf16 (l2_out is BF16 in "Data Flow")
  y_t   = bf16( sum_{j = 0..k-1} w_t,j * bf16(o_{e_j}) )  (in j order)

Readings where the pages are silent:
* The clamp form. "Lucifer-CUTLASS TP3 virtual-padding audit", section
  "TP3 shape plan", gives only swiglu_limit = 10. Reading: the gate is clamped
  above at +L and the up projection is clamped to [-L, L].
* Gate/up order in W13. Rows [0, I) are the gate and rows [I, 2I) are up,
  following "W13 happens to load correctly" (per-half slicing).
* The router bias is an optional additive fp32 term on the logits. It is used
  only to give the Zipf-skewed prefill workload its popularity law.
* Softmax top-k with renormalised weights, as stated for the workloads.
* Moving the expert loop outside the token loop (``moe_tokens``) does not
  change any per-(token, expert) value. The combine still runs in j order per
  token.
"""
from __future__ import annotations

from typing import Callable, NamedTuple

import numpy as np

from . import nvfp4

F32 = np.float32


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


# ---------------------------------------------------------------- routing ----

def router_logits(x_bits: np.ndarray, wr_bits: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """fp32 logits [T, E]: an fp64 dot product rounded once to fp32, then + bias in fp32."""
    l = (bf16_to_f64(x_bits) @ bf16_to_f64(wr_bits).T).astype(F32)
    if bias is not None:
        l = (l + np.asarray(bias, dtype=F32)).astype(F32)
    return l


def topk_softmax(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Top-k ids [T, k] (descending logit, ties to the lower id) and renormalised weights [T, k] fp64."""
    logits = np.asarray(logits, dtype=F32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int64)
    w = np.empty((T, k), dtype=np.float64)
    eidx = np.arange(E)
    for t in range(T):
        order = np.lexsort((eidx, -logits[t]))    # primary: logit descending; secondary: id ascending
        sel = order[:k]
        ids[t] = sel
        l = logits[t, sel].astype(np.float64)
        ex = np.exp(l - l.max())
        w[t] = ex / ex.sum()
    return ids, w


# ---------------------------------------------------------------- experts ----

class QuantExpert(NamedTuple):
    """One expert's NVFP4 weights in logical order (codes unpacked, scales unswizzled)."""
    w1_q: np.ndarray    # [2I, H] codes, rows [0,I) gate, [I,2I) up
    w1_sf: np.ndarray   # [2I, H/16] E4M3
    w1_gs: np.float32   # quant-direction global scale of W1
    w2_q: np.ndarray    # [H, I]
    w2_sf: np.ndarray   # [H, I/16]
    w2_gs: np.float32


def quantize_expert(w1: np.ndarray, w2: np.ndarray) -> QuantExpert:
    """Per-expert, per-matrix global scale from amax, then NVFP4 rows."""
    g1 = nvfp4.global_scale(np.abs(w1).max())
    g2 = nvfp4.global_scale(np.abs(w2).max())
    q1, s1 = nvfp4.quantize_rows(w1, g1)
    q2, s2 = nvfp4.quantize_rows(w2, g2)
    return QuantExpert(q1, s1, g1, q2, s2, g2)


def swiglu(g: np.ndarray, u: np.ndarray, limit: float) -> np.ndarray:
    gc = np.minimum(g, limit)
    uc = np.clip(u, -limit, limit)
    return gc / (1.0 + np.exp(-gc)) * uc


def expert_hidden(qe: QuantExpert, xt: np.ndarray, limit: float) -> np.ndarray:
    """SwiGLU input to the second GEMM, fp64 [n, I], for dequantised activations xt [n, H]."""
    I = qe.w2_q.shape[1]
    W1 = nvfp4.dequantize(qe.w1_q, qe.w1_sf, qe.w1_gs)                  # [2I, H] fp64
    gu = xt @ W1.T                                                      # [n, 2I]
    return swiglu(gu[:, :I], gu[:, I:], limit)


def expert_out(qe: QuantExpert, h: np.ndarray, gs2) -> np.ndarray:
    """Second GEMM of one expert for fp64 hidden rows h [n, I]: requantise, then W2~ h~."""
    q2, s2 = nvfp4.quantize_rows(h.astype(F32), gs2)
    ht = nvfp4.dequantize(q2, s2, gs2)
    W2 = nvfp4.dequantize(qe.w2_q, qe.w2_sf, qe.w2_gs)                  # [H, I]
    return ht @ W2.T


def activation_scale(x_bits: np.ndarray) -> np.float32:
    """gs1 = g(amax |x|) of a warm-up batch ("Current Bug" sections "Bug 5" and "Bug 6")."""
    return nvfp4.global_scale(F32(np.abs(bf16_to_f64(x_bits)).max()))


def dequantized_activations(x_bits: np.ndarray, gs) -> np.ndarray:
    """x~ = dequant(quant(x, gs)) in fp64 [n, H]: the L1 activations every routed expert sees."""
    q, sf = nvfp4.quantize_rows(bf16_to_f64(x_bits).astype(F32), gs)
    return nvfp4.dequantize(q, sf, gs)


def hidden_amax(qe: QuantExpert, xt: np.ndarray, limit: float) -> float:
    """amax |RN_f32(h)| of one expert over dequantised activation rows xt [n, H] (0 for no rows)."""
    if xt.shape[0] == 0:
        return 0.0
    return float(np.abs(expert_hidden(qe, xt, limit).astype(F32)).max())


def pair_rows(qe: QuantExpert, xt: np.ndarray, gs2, limit: float, quantize_activations: bool = True) -> np.ndarray:
    """One expert's W2 output rows o [n, H] (fp64) for dequantised activation rows xt [n, H].

    quantize_activations=False skips the L2 codec (h goes to W2 as it is).
    """
    h = expert_hidden(qe, xt, limit)
    if quantize_activations:
        return expert_out(qe, h, gs2)
    return h @ nvfp4.dequantize(qe.w2_q, qe.w2_sf, qe.w2_gs).T


def routed_rows(ids: np.ndarray) -> dict:
    """expert -> (token rows tt, slots jj) of every routed pair; pairs held by no local expert (-1, "Bug 8") are
    left out."""
    return {int(e): np.nonzero(ids == e) for e in np.unique(ids) if e >= 0}


def l2_out_bf16(outs: np.ndarray) -> np.ndarray:
    """The second GEMM's output as "Data Flow" returns it (l2_out, BF16): fp64 -> fp32 -> bf16, round to nearest
    even at each step, back as fp64."""
    return bf16_to_f64(f32_to_bf16_bits(np.asarray(outs, dtype=np.float64).astype(F32)))


def combine(ids: np.ndarray, w: np.ndarray, outs: np.ndarray, shared: np.ndarray | None = None) -> np.ndarray:
    """y = bf16( sum_{j = 0..k-1} w[:, j] * bf16(outs[:, j]) (+ shared) ), summed in j order; pairs with id -1
    (held elsewhere) are skipped. outs [n, k, H] fp64 are the pair rows of the second GEMM, which "Data Flow"
    returns in BF16 (l2_out) before the scatter_add; shared (fp32 values) is added as it is. Returns bf16
    bits [n, H]."""
    n, k = ids.shape
    outs = l2_out_bf16(outs)
    acc = np.zeros((n, outs.shape[2]), dtype=np.float64)
    for j in range(k):
        held = (ids[:, j] >= 0)[:, None]
        acc = np.where(held, acc + w[:, j:j + 1] * outs[:, j], acc)
    if shared is not None:
        acc = acc + shared
    return f32_to_bf16_bits(acc.astype(F32))


def moe_tokens(x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray,
               expert: Callable[[int], QuantExpert], gs1, gs2, limit: float,
               quantize_activations: bool = True, shared: np.ndarray | None = None) -> np.ndarray:
    """The layer for a set of token rows with their routing. Returns y as bf16 bits [n, H].

    x_bits [n, H] bf16 bits, ids [n, k], w [n, k]. ``expert(e)`` gives the quantised
    weights of expert e. quantize_activations=False replaces both activation
    codecs by the identity (used to pin the layer against a textbook dense MoE).
    ``shared`` [n, H] is a shared expert's output, added with weight 1 after the
    routed terms (``fp8block.shared_out``).
    """
    xt = dequantized_activations(x_bits, gs1) if quantize_activations else bf16_to_f64(x_bits)
    n, H = xt.shape
    outs = np.zeros((n, ids.shape[1], H), dtype=np.float64)
    for e, (tt, jj) in routed_rows(ids).items():
        outs[tt, jj] = pair_rows(expert(e), xt[tt], gs2, limit, quantize_activations)
    return combine(ids, w, outs, shared)


def calibrate(x_bits: np.ndarray, ids: np.ndarray, expert: Callable[[int], QuantExpert], limit: float):
    """Activation global scales from a warmup batch ("Current Bug" sections "Bug 5" and "Bug 6").

    gs1 = g(amax |x|). gs2 = g(amax |h|), taken over every routed (token, expert)
    pair of the warmup batch, with h computed from the gs1-quantised activations.
    With expert parallelism the ids are local and masked pairs (-1) are skipped:
    the fix of "Bug 13", where global ids matched no local expert and gs2 came out 0.
    """
    gs1 = activation_scale(x_bits)
    xt = dequantized_activations(x_bits, gs1)
    amax_h = 0.0
    for e, (tt, _) in routed_rows(ids).items():
        amax_h = max(amax_h, hidden_amax(expert(e), xt[tt], limit))
    return gs1, nvfp4.global_scale(F32(amax_h))
