"""CPU oracle for the top-k consumer of the indexer logits -- TEST
INFRASTRUCTURE ONLY (only tests/, __graft_entry__.smoke() and bench.py's CPU
legs may import it; the product library never does).

The selection that follows the logits on the pages is a per-row top-k
(index_topk 2048 or 512: aiter PR 5047 "GLM-5.2-MXFP4 E2E"; aiter issue 5477,
Measurement).  The pages say no more about it; the definition followed here
(the library's): the k positions of a row's window with the largest logits,
equal logits taken from the lowest positions first (which makes the set
unique; -0.0 equals +0.0), listed in ascending position order and padded
with -1 past the window length.  Plain numpy: a lexicographic sort of each
window, then a sort of the chosen positions.
"""
from __future__ import annotations

import numpy as np


def decode_windows(context_lens, next_n: int, max_model_len: int):
    """Row b*next_n+n: [0, min(ctx_b - next_n + n + 1, max_model_len)) (the
    causal window of the decode logits, aiter PR 5047 Technical Details)."""
    ctx = np.maximum(np.asarray(context_lens, dtype=np.int64), 0)
    b = np.repeat(np.arange(ctx.size), next_n)
    n = np.tile(np.arange(next_n), ctx.size)
    hi = np.minimum(ctx[b] - next_n + n + 1, max_model_len)
    lo = np.zeros_like(hi)
    return lo, np.maximum(hi, lo)


def prefill_windows(ks, ke, width: int):
    """Row m: [max(ks, 0), min(ke, width)) (aiter PR 5046 Motivation, with
    the clamping of its empty / past_end window modes)."""
    lo = np.maximum(np.asarray(ks, dtype=np.int64), 0)
    hi = np.minimum(np.asarray(ke, dtype=np.int64), width)
    return lo, np.maximum(hi, lo)


def topk_rows(logits: np.ndarray, lo, hi, k: int) -> np.ndarray:
    """int32 [rows, k]: per row the first k window positions in (logit desc,
    position asc) order, listed by position, -1 past the window."""
    logits = np.asarray(logits)
    out = np.full((logits.shape[0], k), -1, dtype=np.int32)
    for r in range(logits.shape[0]):
        a, b = int(lo[r]), int(hi[r])
        if b <= a:
            continue
        pos = np.arange(a, b)
        vals = logits[r, a:b].astype(np.float64)  # numeric comparison: -0.0 == +0.0
        order = np.lexsort((pos, -vals))  # last key is primary: value descending, then position
        sel = np.sort(pos[order[:k]])
        out[r, :sel.size] = sel
    return out
