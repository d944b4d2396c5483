"""Pins of the top-k oracle (oracle/topk.py) against values fixed by hand,
library routines and invariants -- not against itself.

The definition (the library's reading of the pages' top-k step): per row,
the k window positions with the largest logits (equal logits: lowest
positions first), listed by position, -1 past the window length; -0.0 equals
+0.0.
"""
import inspect
import textwrap

import numpy as np
import pytest

from oracle import topk as T


def _rows(vals):
    return np.asarray(vals, dtype=np.float32)[None, :]


def pin_hand_cases(topk):
    row = _rows([3, 1, 4, 1, 5, 9, 2, 6])
    full = (np.array([0]), np.array([8]))
    # 9@5 > 6@7 > 5@4 > 4@2 > 3@0 > 2@6 > 1@1 = 1@3 (tie: lower position first)
    assert topk(row, *full, 3).tolist() == [[4, 5, 7]]
    assert topk(row, *full, 7).tolist() == [[0, 1, 2, 4, 5, 6, 7]]  # of the two 1s, position 1
    assert topk(row, *full, 8).tolist() == [[0, 1, 2, 3, 4, 5, 6, 7]]
    # window [2, 6): 4@2, 1@3, 5@4, 9@5
    assert topk(row, np.array([2]), np.array([6]), 3).tolist() == [[2, 4, 5]]
    # window shorter than k: padded with -1
    assert topk(row, np.array([6]), np.array([8]), 4).tolist() == [[6, 7, -1, -1]]
    # empty window
    assert topk(row, np.array([5]), np.array([5]), 2).tolist() == [[-1, -1]]
    # equal values: the lowest positions
    assert topk(_rows([1.0, 5.0, 5.0, 5.0]), np.array([0]), np.array([4]), 2).tolist() == [[1, 2]]
    # -0.0 equals +0.0 (position order decides), -inf is the smallest value
    assert topk(_rows([-1.0, -0.0, 0.0, -0.0]), np.array([0]), np.array([4]), 2).tolist() == [[1, 2]]
    assert topk(_rows([-1.0, 0.0, -0.0, 0.0]), np.array([0]), np.array([4]), 2).tolist() == [[1, 2]]
    assert topk(_rows([-np.inf, 1.0, -np.inf, -np.inf]), np.array([0]), np.array([4]), 2).tolist() == [[0, 1]]


def pin_windows(decode_windows, prefill_windows):
    # ctx 5, next_n 2, max_model_len 4: rows see p <= 5-2+n, capped at 4 columns;
    # ctx 0: p <= -2+n, empty for both rows
    lo, hi = decode_windows([5, 0], 2, 4)
    assert lo.tolist() == [0, 0, 0, 0] and hi.tolist() == [4, 4, 0, 0]
    lo, hi = decode_windows([7], 3, 100)
    assert hi.tolist() == [5, 6, 7]
    # prefill: clamp to [0, width); ke <= ks is empty
    lo, hi = prefill_windows([-3, 2, 9, 4], [5, 12, 20, 4], 10)
    assert lo.tolist() == [0, 2, 9, 4] and hi.tolist() == [5, 10, 10, 4]


def pin_argmax(topk):
    """k = 1 is numpy's argmax over the window (first occurrence on ties)."""
    rng = np.random.default_rng(0)
    logits = np.round(rng.normal(size=(40, 300)), 1).astype(np.float32)  # many exact ties
    lo = rng.integers(0, 150, 40)
    hi = lo + rng.integers(1, 150, 40)
    got = topk(logits, lo, hi, 1)[:, 0]
    want = [lo[r] + int(np.argmax(logits[r, lo[r]:hi[r]])) for r in range(40)]
    assert got.tolist() == want


def pin_partition(topk):
    """Distinct values: the selected set is every window position whose value
    is at least the k-th largest (numpy's partition)."""
    rng = np.random.default_rng(1)
    logits = rng.permutation(np.arange(30 * 500, dtype=np.float32)).reshape(30, 500) / 7.0
    lo = rng.integers(0, 100, 30)
    hi = np.minimum(lo + rng.integers(50, 400, 30), 500)
    for k in (1, 9, 50):
        got = topk(logits, lo, hi, k)
        for r in range(30):
            w = logits[r, lo[r]:hi[r]]
            kk = min(k, w.size)
            kth = np.partition(w, w.size - kk)[w.size - kk]
            assert set(got[r, :kk].tolist()) == set((lo[r] + np.nonzero(w >= kth)[0]).tolist())


def pin_invariants(topk):
    """Position order, uniqueness, window membership, padding; nothing left
    out is larger than anything kept, and at the boundary value the kept
    positions are the lowest ones; doubling every value (exact) changes
    nothing."""
    rng = np.random.default_rng(2)
    logits = np.round(rng.normal(size=(25, 700)) * 4).astype(np.float32)
    lo = rng.integers(0, 300, 25)
    hi = lo + rng.integers(0, 400, 25)
    hi = np.minimum(hi, 700)
    k = 64
    got = topk(logits, lo, hi, k)
    for r in range(25):
        n = int(hi[r] - lo[r])
        sel = got[r, :min(k, n)]
        assert (got[r, min(k, n):] == -1).all()
        assert len(set(sel.tolist())) == sel.size
        assert ((sel >= lo[r]) & (sel < hi[r])).all()
        assert (np.diff(sel) > 0).all()
        if n > k:
            rest = np.setdiff1d(np.arange(lo[r], hi[r]), sel)
            low = logits[r, sel].min()
            assert logits[r, rest].max() <= low
            kept_at_low = sel[logits[r, sel] == low]
            left_at_low = rest[logits[r, rest] == low]
            if left_at_low.size:
                assert kept_at_low.max() < left_at_low.min()
    assert np.array_equal(topk(logits * 2, lo, hi, k), got)


def run_pins(topk=T.topk_rows, decode_windows=T.decode_windows, prefill_windows=T.prefill_windows):
    pin_hand_cases(topk)
    pin_windows(decode_windows, prefill_windows)
    pin_argmax(topk)
    pin_partition(topk)
    pin_invariants(topk)


def test_topk_oracle_pins():
    run_pins()


# Plausible mistakes planted in copies of the oracle; each must fail a pin.
MUTANTS = {
    "ascending": ("np.lexsort((pos, -vals))", "np.lexsort((pos, vals))"),
    "unsorted_output": ("sel = np.sort(pos[order[:k]])", "sel = pos[order[:k]]"),
    "ties_descending": ("np.lexsort((pos, -vals))", "np.lexsort((-pos, -vals))"),
    "raw_bit_order": ("logits[r, a:b].astype(np.float64)", "logits[r, a:b].astype(np.float64).view(np.int64)"),
    "pad_zero": ("np.full((logits.shape[0], k), -1, dtype=np.int32)", "np.zeros((logits.shape[0], k), dtype=np.int32)"),
    "window_end_inclusive": ("a, b = int(lo[r]), int(hi[r])", "a, b = int(lo[r]), int(hi[r]) + 1"),
    "decode_bound_exclusive": ("ctx[b] - next_n + n + 1", "ctx[b] - next_n + n"),
    "decode_no_cap": ("np.minimum(ctx[b] - next_n + n + 1, max_model_len)", "ctx[b] - next_n + n + 1"),
    "prefill_no_clamp": ("np.maximum(np.asarray(ks, dtype=np.int64), 0)", "np.asarray(ks, dtype=np.int64)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_topk_oracle_mutants_fail(name):
    old, new = MUTANTS[name]
    src = inspect.getsource(T)
    assert src.count(old) == 1, name
    ns = {"np": np, "__name__": "mutant"}
    exec(compile(textwrap.dedent(src.replace(old, new)), f"<mutant {name}>", "exec"), ns)
    if name == "window_end_inclusive":
        # the mutant reads one column past the window; give it room
        def topk(logits, lo, hi, k):
            padded = np.concatenate([logits, np.full((logits.shape[0], 1), 1e9, np.float32)], axis=1)
            return ns["topk_rows"](padded, lo, hi, k)
    else:
        topk = ns["topk_rows"]
    with pytest.raises(AssertionError):
        run_pins(topk, ns["decode_windows"], ns["prefill_windows"])
