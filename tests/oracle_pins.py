"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on deliberately broken copies of the
oracle source and requires every copy to fail at least one pin.

What each pin rests on:
  * the e4m3 format definition (OCP OFP8) and an independent library cast;
  * hand-worked cases whose expected values are derived in the comments;
  * a closed form: with non-negative Q and K every ReLU is the identity, so a
    logit row is one matrix-vector product (numpy, on library-decoded values);
  * invariants stated by the indexer pages: the kv_scale hoist (scale >= 0 and
    ReLU positive-homogeneous), linearity in the weights, zero contribution of
    heads whose dot product is negative, exact window placement, block-table
    permutation invariance, decode/prefill consistency.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import workloads

NINF = -math.inf


def lib_decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """e4m3 codes -> float64 via torch's float8_e4m3fn (independent of the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _close(a, b, rtol=1e-12, atol=1e-12):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    fa, fb = np.isfinite(a), np.isfinite(b)
    assert np.array_equal(fa, fb), "finite masks differ"
    assert np.array_equal(a[~fa], b[~fb]), "non-finite values differ"
    if fa.any():
        err = np.abs(a[fa] - b[fb])
        tol = atol + rtol * np.maximum(np.abs(a[fa]), np.abs(b[fb]))
        assert np.all(err <= tol), f"max err {err.max()} (worst tol {tol[err.argmax()]})"


# ---------------------------------------------------------------- e4m3 decode
def pin_e4m3_format(o):
    """Spot values fixed by the OFP8 E4M3 definition (bias 7, no inf)."""
    spot = {
        0x00: 0.0, 0x80: -0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,
        0x08: 2.0 ** -6, 0x38: 1.0, 0x3F: 1.875, 0x40: 2.0, 0x44: 3.0,
        0x30: 0.5, 0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0, 0x77: 240.0,
    }
    for code, val in spot.items():
        got = o.e4m3_to_double(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (hex(code), got, val)
    assert math.isnan(o.e4m3_to_double(0x7F)) and math.isnan(o.e4m3_to_double(0xFF))


def pin_e4m3_all_codes(o):
    """All 256 codes agree with torch's float8_e4m3fn conversion."""
    ref = lib_decode_e4m3(np.arange(256, dtype=np.uint8))
    got = np.array([o.e4m3_to_double(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


# ----------------------------------------------------------- hand-worked cases
def _code(v):
    return int(workloads.e4m3_codes(np.array([v], np.float32))[0])


def pin_hand_prefill(o):
    """H=2, D=128, one query row, two K rows, window [0, 2).

    Q head0: 1.0 @ d0, 2.0 @ d5        Q head1: -1.0 @ d0, 0.5 @ d127
    K row0: 3.0 @ d0, 1.0 @ d5, 2.0 @ d127     K row1: -1.0 @ d0, 448 @ d127
    kv_scale = [0.25, 2.0]; weights = [0.5, -3.0]

    n=0: head0 dot = 1*3 + 2*1 = 5; head1 dot = -3 + 0.5*2 = -2 -> relu 0
         logit = 5 * 0.25 * 0.5 = 0.625
    n=1: head0 dot = -1 -> 0; head1 dot = 1 + 0.5*448 = 225
         logit = 225 * 2.0 * (-3.0) = -1350
    A third row with window [1, 2) sees only n=1 with weights [1, 1]:
         logit = 225 * 2 * 1 = 450, and -inf at n=0.
    """
    q = np.zeros((2, 2, 128), np.uint8)
    q[:, 0, 0] = _code(1.0)
    q[:, 0, 5] = _code(2.0)
    q[:, 1, 0] = _code(-1.0)
    q[:, 1, 127] = _code(0.5)
    k = np.zeros((2, 128), np.uint8)
    k[0, 0], k[0, 5], k[0, 127] = _code(3.0), _code(1.0), _code(2.0)
    k[1, 0], k[1, 127] = _code(-1.0), _code(448.0)
    s = np.array([0.25, 2.0], np.float32)
    w = np.array([[0.5, -3.0], [1.0, 1.0]], np.float32)
    ks = np.array([0, 1], np.int32)
    ke = np.array([2, 2], np.int32)
    out = o.mqa_logits(q, k, s, w, ks, ke)
    _close(out, [[0.625, -1350.0], [NINF, 450.0]], rtol=0, atol=0)


def hand_decode_inputs():
    """B=1, next_n=2, H=1, D=128, block_size=2, ctx=3, max_model_len=4.

    Tokens: t0 = 2.0 @ d3 (scale 1.0); t1 = 1.0 @ d3, 1.0 @ d4 (scale 0.5);
            t2 = -2.0 @ d3 (scale 4.0).
    Physical blocks are swapped: block_tables = [[1, 0]], so t0, t1 live in
    block 1 (slots 0, 1) and t2 in block 0 slot 0; block 0 slot 1 is unowned
    and NaN-poisoned.
    Q row0 (n=0): 1.0 @ d3, weight 2.0;  Q row1 (n=1): 1.0 @ d3, 3.0 @ d4,
    weight 0.25.
    Windows: row0 p <= 3-2+0 = 1; row1 p <= 2.
      row0: p0 dot 2 -> 2*1*2 = 4;  p1 dot 1 -> 1*0.5*2 = 1
      row1: p0 dot 2 -> 2*1*0.25 = 0.5; p1 dot 1+3 = 4 -> 4*0.5*0.25 = 0.5;
            p2 dot -2 -> 0
    """
    bs, d = 2, 128
    cache = np.zeros((2, bs * (d + 4)), np.uint8)
    kpart = cache[:, : bs * d].reshape(2, bs, d)
    spart = cache[:, bs * d:].view(np.float32).reshape(2, bs)
    kpart[1, 0, 3] = _code(2.0)
    kpart[1, 1, 3] = _code(1.0)
    kpart[1, 1, 4] = _code(1.0)
    kpart[0, 0, 3] = _code(-2.0)
    kpart[0, 1, :] = 0x7F
    spart[1] = [1.0, 0.5]
    spart[0] = [4.0, np.nan]
    q = np.zeros((1, 2, 1, d), np.uint8)
    q[0, 0, 0, 3] = _code(1.0)
    q[0, 1, 0, 3] = _code(1.0)
    q[0, 1, 0, 4] = _code(3.0)
    w = np.array([[2.0], [0.25]], np.float32)
    return dict(q=q, kv_cache=cache, weights=w,
                context_lens=np.array([3], np.int32),
                block_tables=np.array([[1, 0]], np.int32),
                block_size=bs, max_model_len=4)


def pin_hand_decode(o):
    out = o.paged_mqa_logits(**hand_decode_inputs())
    _close(out, [[4.0, 1.0, NINF, NINF], [0.5, 0.5, 0.0, NINF]], rtol=0, atol=0)


# ------------------------------------------------------------------ closed form
def _nonneg(codes):
    return (codes & 0x7F).astype(np.uint8)  # clear the sign bit


def pin_closed_form_prefill(o):
    """Non-negative Q, K: logit[m, n] = s_n * <sum_h w[m,h] Q[m,h,:], K[n,:]>."""
    c = workloads.prefill_case(7, 40, 5, mode="causal", seed=11)
    q, k = _nonneg(c.q), _nonneg(c.k)
    ks = np.zeros(7, np.int32)
    ke = np.full(7, 40, np.int32)
    out = o.mqa_logits(q, k, c.kv_scale, c.weights, ks, ke)
    qd = lib_decode_e4m3(q)              # [M, H, D]
    kd = lib_decode_e4m3(k)              # [N, D]
    w = c.weights.astype(np.float64)     # [M, H]
    qw = np.einsum("mh,mhd->md", w, qd)  # [M, D]
    ref = (qw @ kd.T) * c.kv_scale.astype(np.float64)[None, :]
    _close(out, ref, rtol=1e-12, atol=1e-9)


def pin_closed_form_decode(o):
    c = workloads.decode_case(3, 3, 6, max_model_len=150, block_size=8,
                              var_ratio=0.3, seed=12, extra_blocks=3)
    q = _nonneg(c.q)
    cache = c.kv_cache.copy()
    bs, d = c.block_size, c.dim
    cache[:, : bs * d] &= 0x7F
    out = o.paged_mqa_logits(q, cache, c.weights, c.context_lens,
                             c.block_tables, bs, c.max_model_len)
    qd = lib_decode_e4m3(q)  # [B, next_n, H, D]
    for b in range(c.batch):
        ctx = int(c.context_lens[b])
        toks = np.arange(ctx)
        pages = c.block_tables[b, toks // bs]
        slots = toks % bs
        krow = cache[:, : bs * d].reshape(-1, bs, d)[pages, slots]       # [ctx, D]
        scl = cache[:, bs * d:].view(np.float32).reshape(-1, bs)[pages, slots]
        kd = lib_decode_e4m3(krow)
        for n in range(c.next_n):
            r = b * c.next_n + n
            qw = (c.weights[r].astype(np.float64)[:, None] * qd[b, n]).sum(0)
            ref = np.full(c.max_model_len, NINF)
            last = ctx - c.next_n + n
            ref[: last + 1] = (kd[: last + 1] @ qw) * scl[: last + 1].astype(np.float64)
            _close(out[r], ref, rtol=1e-12, atol=1e-9)


# ------------------------------------------------------------------- invariants
def pin_kv_scale_hoist(o):
    """Positive homogeneity: doubling K exactly equals doubling the scale, and
    the scale factors out of the head sum."""
    c = workloads.prefill_case(6, 33, 4, mode="causal", seed=13)
    kd = lib_decode_e4m3(c.k)
    small = np.abs(kd) <= 224  # doubling stays representable and exact
    k = np.where(small, c.k, 0).astype(np.uint8)
    k2 = workloads.e4m3_codes(2.0 * lib_decode_e4m3(k).astype(np.float32))
    assert np.array_equal(lib_decode_e4m3(k2), 2.0 * lib_decode_e4m3(k))
    ks = np.zeros(6, np.int32)
    ke = np.full(6, 33, np.int32)
    a = o.mqa_logits(c.q, k2, c.kv_scale, c.weights, ks, ke)
    b = o.mqa_logits(c.q, k, 2.0 * c.kv_scale, c.weights, ks, ke)
    _close(a, b, rtol=1e-13, atol=1e-12)
    one = o.mqa_logits(c.q, k, np.ones(33, np.float32), c.weights, ks, ke)
    _close(b, one * (2.0 * c.kv_scale.astype(np.float64))[None, :], rtol=1e-13, atol=1e-12)


def pin_linearity_in_weights(o):
    c = workloads.prefill_case(5, 30, 4, mode="causal", seed=14)
    rng = np.random.default_rng(5)
    # small dyadic values, so alpha*w1 + beta*w2 is exact in f32
    w1 = (rng.integers(-64, 65, c.weights.shape) / 8.0).astype(np.float32)
    w2 = (rng.integers(-64, 65, c.weights.shape) / 8.0).astype(np.float32)
    alpha, beta = 0.5, -2.0
    wc = (alpha * w1 + beta * w2).astype(np.float32)
    assert np.array_equal(wc.astype(np.float64), alpha * w1.astype(np.float64) + beta * w2.astype(np.float64))
    ks = np.zeros(5, np.int32)  # full windows: no -inf to combine
    ke = np.full(5, 30, np.int32)
    f = lambda w: o.mqa_logits(c.q, c.k, c.kv_scale, w, ks, ke)
    _close(f(wc), alpha * f(w1) + beta * f(w2), rtol=1e-12, atol=1e-9)


def pin_negative_heads_contribute_zero(o):
    """Changing the weight of any head whose dot is negative changes nothing;
    changing a head whose dot is positive does change the logit."""
    c = workloads.prefill_case(8, 1, 6, mode="causal", seed=15)
    ks = np.zeros(8, np.int32)
    ke = np.ones(8, np.int32)
    dots = np.einsum("mhd,d->mh", lib_decode_e4m3(c.q), lib_decode_e4m3(c.k[0]))
    assert (dots < 0).any() and (dots > 0).any()
    base = o.mqa_logits(c.q, c.k, c.kv_scale, c.weights, ks, ke)
    w = c.weights.copy()
    w[dots < 0] = 1000.0
    _close(o.mqa_logits(c.q, c.k, c.kv_scale, w, ks, ke), base, rtol=0, atol=0)
    w = c.weights.copy()
    w[dots > 0] += 1.0
    changed = o.mqa_logits(c.q, c.k, c.kv_scale, w, ks, ke)
    rows = (dots > 0).any(axis=1)
    assert np.all(changed[rows, 0] != base[rows, 0])


def pin_decode_window_placement(o):
    """Finite exactly on p <= ctx - next_n + n (and p < max_model_len)."""
    c = workloads.decode_case(4, 3, 2, max_model_len=100, block_size=4,
                              context_lens=[100, 1, 2, 57], seed=16)
    out = o.paged_mqa_logits(c.q, c.kv_cache, c.weights, c.context_lens,
                             c.block_tables, c.block_size, c.max_model_len)
    expect_count = {(0, 0): 98, (0, 1): 99, (0, 2): 100, (1, 0): 0, (1, 1): 0,
                    (1, 2): 1, (2, 0): 0, (2, 1): 1, (2, 2): 2, (3, 0): 55,
                    (3, 1): 56, (3, 2): 57}
    for (b, n), cnt in expect_count.items():
        row = out[b * 3 + n]
        fin = np.isfinite(row)
        assert fin[:cnt].all() and not fin[cnt:].any(), (b, n, fin.sum(), cnt)
        assert np.all(row[cnt:] == NINF)


def pin_block_table_invariance(o):
    """Permuting physical blocks with the table, and NaN-poisoning unowned
    blocks and tail slots, leaves every output unchanged."""
    kw = dict(max_model_len=90, block_size=8, context_lens=[90, 37, 61], seed=17)
    c = workloads.decode_case(3, 2, 3, extra_blocks=4, **kw)
    p = workloads.decode_case(3, 2, 3, extra_blocks=4, poison=True, **kw)
    base = o.paged_mqa_logits(c.q, c.kv_cache, c.weights, c.context_lens,
                              c.block_tables, 8, 90)
    poisoned = o.paged_mqa_logits(p.q, p.kv_cache, p.weights, p.context_lens,
                                  p.block_tables, 8, 90)
    _close(poisoned, base, rtol=0, atol=0)
    rng = np.random.default_rng(3)
    perm = rng.permutation(c.kv_cache.shape[0])       # new position of block i
    cache2 = np.empty_like(c.kv_cache)
    cache2[perm] = c.kv_cache
    tab2 = np.where(c.block_tables >= 0, perm[np.maximum(c.block_tables, 0)], -1).astype(np.int32)
    moved = o.paged_mqa_logits(c.q, cache2, c.weights, c.context_lens, tab2, 8, 90)
    _close(moved, base, rtol=0, atol=0)


def pin_decode_matches_prefill(o):
    """Decode row (b, n) equals the prefill formula on the gathered K with the
    window [0, ctx - next_n + n + 1)."""
    c = workloads.decode_case(2, 3, 4, max_model_len=70, block_size=16,
                              context_lens=[70, 45], seed=18, extra_blocks=2)
    out = o.paged_mqa_logits(c.q, c.kv_cache, c.weights, c.context_lens,
                             c.block_tables, 16, 70)
    d = c.dim
    kp = c.kv_cache[:, : 16 * d].reshape(-1, 16, d)
    sp = c.kv_cache[:, 16 * d:].view(np.float32).reshape(-1, 16)
    for b in range(2):
        ctx = int(c.context_lens[b])
        t = np.arange(ctx)
        kb = kp[c.block_tables[b, t // 16], t % 16]
        sb = sp[c.block_tables[b, t // 16], t % 16]
        q = c.q[b]                                    # [next_n, H, D]
        w = c.weights[b * 3:(b + 1) * 3]
        ks = np.zeros(3, np.int32)
        ke = np.array([ctx - 3 + n + 1 for n in range(3)], np.int32)
        pre = o.mqa_logits(q, kb, sb, w, ks, ke)      # [3, ctx]
        ref = np.full((3, 70), NINF)
        ref[:, :ctx] = pre
        _close(out[b * 3:(b + 1) * 3], ref, rtol=0, atol=0)


def pin_prefill_window_modes(o):
    """-inf exactly outside [max(ks, 0), min(ke, N)) for every window mode."""
    for mode in ("causal", "multi_req", "misaligned", "empty", "past_end", "cp"):
        c = workloads.prefill_case(12, 96, 2, mode=mode, seed=19)
        out = o.mqa_logits(c.q, c.k, c.kv_scale, c.weights, c.ks, c.ke)
        n = np.arange(96)[None, :]
        lo = np.maximum(c.ks.astype(np.int64), 0)[:, None]
        hi = np.minimum(c.ke.astype(np.int64), 96)[:, None]
        inside = (n >= lo) & (n < hi)
        assert np.array_equal(np.isfinite(out), inside), mode
        assert np.all(out[~inside] == NINF), mode


def pin_sampled_matches_dense(o):
    """The element-wise entry points agree with the dense ones."""
    c = workloads.decode_case(2, 2, 3, max_model_len=40, block_size=4,
                              context_lens=[40, 23], seed=20)
    dense = o.paged_mqa_logits(c.q, c.kv_cache, c.weights, c.context_lens,
                               c.block_tables, 4, 40)
    rows, cols = np.meshgrid(np.arange(4), np.arange(40), indexing="ij")
    at = o.paged_mqa_logits_at(c.q, c.kv_cache, c.weights, c.context_lens,
                               c.block_tables, 4, 40, rows.ravel(), cols.ravel())
    _close(at.reshape(4, 40), dense, rtol=0, atol=0)
    p = workloads.prefill_case(5, 17, 2, mode="past_end", seed=21)
    dense = o.mqa_logits(p.q, p.k, p.kv_scale, p.weights, p.ks, p.ke)
    rows, cols = np.meshgrid(np.arange(5), np.arange(17), indexing="ij")
    at = o.mqa_logits_at(p.q, p.k, p.kv_scale, p.weights, p.ks, p.ke,
                         rows.ravel(), cols.ravel())
    _close(at.reshape(5, 17), dense, rtol=0, atol=0)


ALL_PINS = [
    pin_e4m3_format, pin_e4m3_all_codes, pin_hand_prefill, pin_hand_decode,
    pin_closed_form_prefill, pin_closed_form_decode, pin_kv_scale_hoist,
    pin_linearity_in_weights, pin_negative_heads_contribute_zero,
    pin_decode_window_placement, pin_block_table_invariance,
    pin_decode_matches_prefill, pin_prefill_window_modes,
    pin_sampled_matches_dense,
]
