"""Pins of the oracle's counts / offsets / slot layout / capacity."""
import json
import os

import numpy as np
import torch

from oracle import layout

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "runner_bug_history.json")))


def test_offsets_have_no_leading_zero():
    g = GOLD["bug4_offsets"]
    off = layout.inclusive_offsets(np.array(g["counts"]))
    assert list(off) == g["offsets_no_leading_zero"]
    assert list(off) != g["offsets_wrong_with_leading_zero"]
    # torch.cumsum is the library statement of an inclusive running sum
    assert list(off) == torch.cumsum(torch.tensor(g["counts"]), 0).tolist()


def test_searchsorted_right_assigns_row_4_to_expert_1():
    g = GOLD["bug2_searchsorted"]
    off = np.array(g["offsets"])
    assert layout.searchsorted_right(off, g["row"]) == g["right_true"]
    assert layout.searchsorted_left(off, g["row"]) == g["right_false"]
    rng = np.random.default_rng(0)
    for _ in range(50):
        off = np.cumsum(rng.integers(0, 5, 9))
        for row in range(int(off[-1]) + 2):
            ref = int(torch.searchsorted(torch.tensor(off), row, right=True))
            assert layout.searchsorted_right(off, row) == ref


def test_fixed_128_row_slots_overflow_at_prefill():
    g = GOLD["bug9_capacity"]
    assert g["num_experts_fixed_slots"] * g["slot_rows"] == g["fixed_rows"]
    assert g["tokens"] * g["top_k"] == g["pairs"]
    assert g["fixed_rows"] < g["pairs"]
    assert layout.capacity_rows(g["tokens"], g["top_k"], 256) >= g["pairs"]


def test_capacity_bounds_every_padded_layout():
    rng = np.random.default_rng(1)
    for T, k, E in [(1, 6, 256), (2, 2, 8), (16, 2, 8), (21, 6, 256), (64, 6, 256), (512, 6, 256), (8192, 6, 256)]:
        cap = layout.capacity_rows(T, k, E)
        assert cap % 128 == 0 and cap >= 128
        pairs = T * k
        # worst case: as many experts as possible, each with c = 1 (mod 128)
        n = min(E, pairs)
        worst = [1] * n
        worst[0] += pairs - n
        worst += [0] * (E - n)
        assert layout.padded_counts(np.array(worst)).sum() <= cap
        for _ in range(20):
            ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]) if T <= 512 else rng.integers(0, E, (T, k))
            R = layout.slots(ids, E)["R"]
            assert R <= cap
    # T*k <= 128: one 128-row slot per expert is enough
    assert layout.capacity_rows(21, 6, 256) <= 256 * 128


def test_slots_against_stable_sort():
    rng = np.random.default_rng(2)
    for T, k, E in [(16, 2, 8), (64, 6, 256), (300, 6, 16)]:
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
        L = layout.slots(ids, E)
        flat = ids.reshape(-1)
        order = np.argsort(flat, kind="stable")            # pairs grouped by expert, ascending p
        c = np.bincount(flat, minlength=E)
        start = np.concatenate([[0], np.cumsum((c + 127) // 128 * 128)[:-1]])
        rank = np.empty(len(flat), dtype=np.int64)
        seen = {}
        for p in order:
            e = flat[p]
            rank[p] = seen.get(e, 0)
            seen[e] = rank[p] + 1
        assert (L["slot_of_pair"] == start[flat] + rank).all()
        assert (L["counts"] == c).all()
        por = L["pair_of_row"]
        assert (por[L["slot_of_pair"]] == np.arange(len(flat))).all()
        assert (por >= 0).sum() == len(flat)
        # each expert's block starts on a 128-row boundary and holds its rows first
        for e in range(E):
            s = int(L["padded_offsets"][e]) - (int(c[e]) + 127) // 128 * 128
            assert s % 128 == 0
            assert (por[s:s + c[e]] >= 0).all()
            assert (por[s + c[e]: int(L["padded_offsets"][e])] == -1).all()
        # row -> expert through searchsorted(right=True) on the padded ends
        for r in range(0, L["R"], 37):
            e = layout.searchsorted_right(L["padded_offsets"], r)
            if por[r] >= 0:
                assert flat[por[r]] == e


def test_expert_parallel_remap_and_mask():
    """"Bug 8": global ids -> local ids for the held experts, the rest masked; the masked layout is the layout
    of the held pairs alone, and every pair is held by exactly one rank of an EP split."""
    rng = np.random.default_rng(8)
    E, k, T = 256, 6, 40
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    first, count = 96, 48
    loc = layout.local_ids(ids, first, count)
    held = (ids >= first) & (ids < first + count)
    assert (loc[held] == ids[held] - first).all() and (loc[~held] == -1).all()
    L = layout.slots(loc, count)
    flat = loc.reshape(-1)
    assert (L["slot_of_pair"][flat < 0] == -1).all()
    assert L["counts"].sum() == held.sum()
    # the held pairs alone, in pair order, give the same rows
    keep = np.nonzero(flat >= 0)[0]
    L2 = layout.slots(flat[keep], count)
    assert (L["counts"] == L2["counts"]).all() and (L["padded_offsets"] == L2["padded_offsets"]).all()
    assert (L["slot_of_pair"][keep] == L2["slot_of_pair"]).all()
    assert (L["pair_of_row"][L["pair_of_row"] >= 0] == keep[L2["pair_of_row"][L2["pair_of_row"] >= 0]]).all()
    # an 8-way split holds every pair once
    owners = sum((layout.local_ids(ids, 32 * r, 32) >= 0).astype(int) for r in range(8))
    assert (owners == 1).all()
