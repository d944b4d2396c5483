"""Helpers for GPU-vs-oracle parity tests.

Tolerance (from the accuracy bar of the indexer logits): every finite logit
must satisfy |gpu - oracle| <= 1e-3 * max|finite oracle logit of its row|
+ 1e-5, and the set of written / -inf positions must match exactly.  The
oracle is exact (fp64, exact e4m3 products); the GPU accumulates the 128-term
dot products in f32 on the tensor cores and the head sum in f32, so its error
is a few ulps of the largest head term -- far inside the bar.

Also reported (not gated): the pages' calc_diff metric,
1 - 2<x,y> / (<x,x> + <y,y>), which must stay below 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

REL = 1e-3
ABS = 1e-5


def to_device(case, device="cuda"):
    """numpy arrays of a Decode/Prefill case -> torch tensors on the GPU."""
    out = {}
    for k, v in vars(case).items():
        if isinstance(v, np.ndarray):
            out[k] = torch.from_numpy(np.ascontiguousarray(v)).to(device)
    return out


def calc_diff(x: np.ndarray, y: np.ndarray) -> float:
    x = x.astype(np.float64)
    y = y.astype(np.float64)
    den = (x * x).sum() + (y * y).sum()
    if den == 0:
        return 0.0
    return float(1.0 - 2.0 * (x * y).sum() / den)


def assert_rows_close(gpu: np.ndarray, ref: np.ndarray, written: np.ndarray | None = None, what: str = ""):
    """gpu: float32 [R, C]; ref: float64 [R, C] (-inf outside windows).

    written: boolean mask of positions the kernel must write; elsewhere the
    GPU buffer must still hold its NaN poison.  None = every position must be
    written (prefill), with -inf exactly where the oracle has -inf.
    """
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    fin = np.isfinite(ref)
    if written is not None:
        assert np.array_equal(written, fin), f"{what}: oracle window differs from the expected window"
        untouched = np.isnan(gpu)
        bad = untouched == written
        assert not bad.any(), (f"{what}: {int((bad & written).sum())} window positions not written, "
                               f"{int((bad & ~written).sum())} positions outside the window written")
    else:
        ninf_ok = np.array_equal(np.isneginf(gpu), ~fin)
        assert ninf_ok, (f"{what}: -inf mask mismatch: {int((np.isneginf(gpu) & fin).sum())} extra, "
                         f"{int((~np.isneginf(gpu) & ~fin).sum())} missing")
    assert np.isfinite(gpu[fin]).all(), f"{what}: non-finite logits inside windows"
    rowmax = np.where(fin, np.abs(ref), 0.0).max(axis=1, initial=0.0)
    tol = REL * rowmax[:, None] + ABS
    err = np.where(fin, np.abs(gpu.astype(np.float64) - np.where(fin, ref, 0.0)), 0.0)
    worst = err - tol
    if (worst > 0).any():
        r, c = np.unravel_index(np.argmax(worst), worst.shape)
        raise AssertionError(f"{what}: {int((worst > 0).sum())} logits out of tolerance; worst at "
                             f"({r}, {c}): gpu {gpu[r, c]!r} oracle {ref[r, c]!r} tol {tol[r, 0]:.3g}")
    if fin.any():
        cd = calc_diff(gpu[fin], ref[fin])
        assert cd < 1e-3, f"{what}: calc_diff {cd}"


def decode_window_mask(case, rows=None) -> np.ndarray:
    """Boolean [rows, max_model_len]: p <= ctx_b - next_n + n and p < max_model_len."""
    nrows = case.batch * case.next_n
    r0, r1 = (0, nrows) if rows is None else rows
    r = np.arange(r0, r1)
    b = r // case.next_n
    n = r % case.next_n
    last = case.context_lens.astype(np.int64)[b] - case.next_n + n
    p = np.arange(case.max_model_len)[None, :]
    return p <= last[:, None]
