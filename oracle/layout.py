"""Per-expert counts, offsets, 128-row padded slots and their inverse map.

Definitions and the bugs they pin, from "Current Bug: CuTeDSLMoERunner":

* Counts c_e = #{(t, j) : topk_ids[t, j] = e} (section "Bug 4" and the
  device-side counts of "CUDA-Graph Safety", SECTION B: scatter_add_ into a
  preallocated buffer, no bincount).
* Expert offsets are the inclusive cumulative sum WITHOUT a leading 0. Counts
  [4, 4, 0] give [4, 8, 8], not [0, 4, 8, 8] ("Bug 4").
* Row -> expert is searchsorted(offsets, row, right=True). With right=False,
  row 4 of [4, 8, 8] goes wrongly to expert 0 ("Bug 2").
* Each expert's rows start on a 128-row boundary. Padding rows carry nothing
  and are dropped at the combine ("Bug 14").
  P_e = align_up(c_e, 128). Padded offsets are the inclusive sum of P_e,
  also without a leading 0. ("Bug 14" prints [0, 128, 256, ...] with a
  leading 0, which contradicts "Bug 4". Reading: no leading 0 in either array.)
* Slot order inside an expert is ascending pair index p = t*k + j. The pages
  say "sort by expert" with no secondary key; this is the plain stable reading.
* Capacity. A fixed 128 rows per expert overflows at prefill: 48*128 < 8192*6
  ("Bug 9"). The buffers therefore hold
  CAP(T) = align_down(T*k + 127*min(E, T*k), 128), with a floor of 128. That
  bounds sum_e P_e, because each non-empty expert adds at most 127 padding rows.
"""
from __future__ import annotations

import numpy as np

ROW_ALIGN = 128


def align_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def capacity_rows(T: int, k: int, E: int) -> int:
    pairs = T * k
    cap = (pairs + 127 * min(E, pairs)) // ROW_ALIGN * ROW_ALIGN
    return max(cap, ROW_ALIGN)


def local_ids(topk_ids: np.ndarray, first: int, count: int) -> np.ndarray:
    """Expert parallelism ("Current Bug", "Bug 8"): the router's global expert ids become local ids
    id - first for the experts [first, first + count) this layer holds, and -1 (masked out) otherwise."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    local = ids - first
    return np.where((local >= 0) & (local < count), local, -1)


def counts(topk_ids: np.ndarray, E: int) -> np.ndarray:
    """Pairs per expert; masked pairs (id -1) count for none."""
    c = np.zeros(E, dtype=np.int64)
    for e in np.asarray(topk_ids).reshape(-1):
        if e >= 0:
            c[int(e)] += 1
    return c


def inclusive_offsets(c: np.ndarray) -> np.ndarray:
    """Inclusive running sum, no leading zero."""
    out = np.zeros(len(c), dtype=np.int64)
    run = 0
    for e, v in enumerate(c):
        run += int(v)
        out[e] = run
    return out


def padded_counts(c: np.ndarray) -> np.ndarray:
    return np.array([align_up(int(v), ROW_ALIGN) for v in c], dtype=np.int64)


def searchsorted_right(offsets: np.ndarray, row: int) -> int:
    """Number of entries <= row, i.e. the expert that owns ``row`` given inclusive ends."""
    n = 0
    for v in offsets:
        if v <= row:
            n += 1
    return n


def searchsorted_left(offsets: np.ndarray, row: int) -> int:
    n = 0
    for v in offsets:
        if v < row:
            n += 1
    return n


def slots(topk_ids: np.ndarray, E: int):
    """The full padded layout of a routing decision.

    Returns a dict with:
      counts, offsets, padded_offsets : [E] int64
      slot_of_pair                    : [T*k] int64, -1 for a masked pair (id -1)
      pair_of_row                     : [R] int64, -1 on padding rows (R = padded_offsets[-1])
    """
    ids = np.asarray(topk_ids).reshape(-1)
    c = counts(ids, E)
    off = inclusive_offsets(c)
    P = padded_counts(c)
    poff = inclusive_offsets(P)
    R = int(poff[-1]) if E > 0 else 0
    seen = np.zeros(E, dtype=np.int64)
    slot = np.zeros(len(ids), dtype=np.int64)
    for p, e in enumerate(ids):
        e = int(e)
        if e < 0:
            slot[p] = -1
            continue
        slot[p] = (poff[e] - P[e]) + seen[e]
        seen[e] += 1
    pair_of_row = np.full(R, -1, dtype=np.int64)
    held = slot >= 0
    pair_of_row[slot[held]] = np.arange(len(ids))[held]
    return dict(counts=c, offsets=off, padded_offsets=poff, slot_of_pair=slot, pair_of_row=pair_of_row, R=R)
