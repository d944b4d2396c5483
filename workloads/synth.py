"""Seeded synthetic workloads for the indexer logits.

Value recipe (the benchmark configurations of the indexer pages, restated):
  * Q ~ N(0, 1), cast to e4m3 (round-to-nearest-even, clamped to +-448).
  * K ~ N(0, 1) per token; per-token scale = max(amax, 1e-4) / 448; K is
    stored as e4m3(clamp(K / scale, +-448)).  The 1e-4 guard only matters for
    an all-zero row.
  * weights ~ N(0, 1) / sqrt(32), f32 (the same divisor for every head count).
  * ragged contexts: ctx = floor(L * (1 - U(0, var_ratio))), at least next_n.

Decode cache layout ("split page"): kv_cache is [num_blocks, block_size*(D+4)]
bytes; a block holds block_size K rows of D e4m3 bytes followed by block_size
f32 scales.  Block size 1 is the plain co-packed cache: D K bytes, then the
4-byte scale, per token.  Physical blocks are a seeded permutation of the
pool, so walking the cache linearly gives wrong answers.

No logits arithmetic lives here: only random draws, casts and layout.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

E4M3_MAX = 448.0
NAN_CODE = 0x7F  # S.1111.111 is NaN in e4m3


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 array -> uint8 e4m3 codes (RNE, clamped to +-448)."""
    x = np.clip(np.asarray(x, dtype=np.float32), -E4M3_MAX, E4M3_MAX)
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _k_tokens(rng: np.random.Generator, n: int, dim: int):
    """n K rows: (codes [n, dim] u8, scale [n] f32) per the value recipe."""
    k = rng.standard_normal((n, dim), dtype=np.float32)
    amax = np.abs(k).max(axis=1) if n else np.zeros((0,), np.float32)
    scale = (np.maximum(amax, np.float32(1e-4)) / np.float32(E4M3_MAX)).astype(np.float32)
    codes = e4m3_codes(k / scale[:, None]) if n else np.zeros((0, dim), np.uint8)
    return codes, scale


def _q_codes(rng, shape):
    return e4m3_codes(rng.standard_normal(shape, dtype=np.float32))


def _weights(rng, rows, heads):
    w = rng.standard_normal((rows, heads), dtype=np.float32) / np.float32(math.sqrt(32.0))
    return w.astype(np.float32)


@dataclasses.dataclass
class DecodeCase:
    q: np.ndarray             # [B, next_n, H, D] u8 (e4m3)
    kv_cache: np.ndarray      # [num_blocks, block_size*(D+4)] u8
    weights: np.ndarray       # [B*next_n, H] f32
    context_lens: np.ndarray  # [B] i32
    block_tables: np.ndarray  # [B, max_blocks] i32
    block_size: int
    max_model_len: int
    name: str = ""

    @property
    def batch(self):
        return self.q.shape[0]

    @property
    def next_n(self):
        return self.q.shape[1]

    @property
    def heads(self):
        return self.q.shape[2]

    @property
    def dim(self):
        return self.q.shape[3]

    def owned_positions(self) -> int:
        """Number of written output elements (sum of window lengths)."""
        tot = 0
        for c in self.context_lens.tolist():
            for n in range(self.next_n):
                last = min(c - self.next_n + n, self.max_model_len - 1)
                tot += max(0, last + 1)
        return tot


def decode_case(batch, next_n, heads, dim=128, max_model_len=1024,
                block_size=64, context_lens=None, var_ratio=0.0, seed=0,
                poison=False, extra_blocks=0, table_fill=-1, name=""):
    """Build one seeded decode workload.

    context_lens: explicit list, or None for floor(L*(1-U(0,var_ratio))) with
    L = max_model_len.  poison=True fills unowned blocks and the tail slots of
    the last block of each request with NaN codes / NaN scales.
    extra_blocks adds unowned blocks to the pool.  Unused block-table entries
    hold table_fill.
    """
    rng = np.random.default_rng(seed)
    if context_lens is None:
        u = rng.uniform(0.0, var_ratio, size=batch) if var_ratio > 0 else np.zeros(batch)
        ctx = np.floor(max_model_len * (1.0 - u)).astype(np.int64)
        ctx = np.maximum(ctx, next_n)
    else:
        ctx = np.asarray(context_lens, dtype=np.int64)
    assert ctx.shape == (batch,)
    max_blocks = -(-max_model_len // block_size)
    blocks_per_req = [max(0, -(-int(c) // block_size)) for c in ctx]
    owned = sum(blocks_per_req)
    pool = owned + extra_blocks
    perm = rng.permutation(pool).astype(np.int32)

    q = _q_codes(rng, (batch, next_n, heads, dim))
    w = _weights(rng, batch * next_n, heads)

    page_bytes = block_size * (dim + 4)
    if poison:
        cache = np.full((pool, page_bytes), NAN_CODE, np.uint8)
        # NaN f32 scales in every slot: bytes 0x7F 0xC0 0x00 0x00 little-endian
        scales_view = cache[:, block_size * dim:].view(np.uint32)
        scales_view[:] = np.uint32(0x7FC00000)
    else:
        cache = np.zeros((pool, page_bytes), np.uint8)
    tables = np.full((batch, max_blocks), table_fill, np.int32)
    k_part = cache[:, : block_size * dim].reshape(pool, block_size, dim)
    s_part = cache[:, block_size * dim:].view(np.float32).reshape(pool, block_size)

    nxt = 0
    for b in range(batch):
        c = int(ctx[b])
        nb = blocks_per_req[b]
        ids = perm[nxt: nxt + nb]
        nxt += nb
        tables[b, :nb] = ids
        if c <= 0:
            continue
        codes, scale = _k_tokens(rng, c, dim)
        full = c // block_size
        if full:
            k_part[ids[:full]] = codes[: full * block_size].reshape(full, block_size, dim)
            s_part[ids[:full]] = scale[: full * block_size].reshape(full, block_size)
        tail = c - full * block_size
        if tail:
            k_part[ids[full], :tail] = codes[full * block_size:]
            s_part[ids[full], :tail] = scale[full * block_size:]
    return DecodeCase(q=q, kv_cache=cache, weights=w,
                      context_lens=ctx.astype(np.int32), block_tables=tables,
                      block_size=block_size, max_model_len=max_model_len,
                      name=name)


@dataclasses.dataclass
class PrefillCase:
    q: np.ndarray         # [M, H, D] u8
    k: np.ndarray         # [N, D] u8
    kv_scale: np.ndarray  # [N] f32
    weights: np.ndarray   # [M, H] f32
    ks: np.ndarray        # [M] i32
    ke: np.ndarray        # [M] i32
    name: str = ""

    @property
    def rows(self):
        return self.q.shape[0]

    @property
    def cols(self):
        return self.k.shape[0]

    @property
    def heads(self):
        return self.q.shape[1]

    def window_pairs(self) -> int:
        lo = np.maximum(self.ks.astype(np.int64), 0)
        hi = np.minimum(self.ke.astype(np.int64), self.cols)
        return int(np.maximum(hi - lo, 0).sum())


def prefill_windows(mode: str, m: int, n: int, rng: np.random.Generator,
                    requests: int = 4):
    """Per-row [ks, ke) windows for the prefill window modes.

    causal    one request; its M rows are the last M of N positions.
    multi_req `requests` packed requests, each owning N/requests K tokens
              with its rows the last rows of that range; request sizes are
              uneven so row blocks straddle request boundaries.
    misaligned like causal but the request starts at an odd K offset.
    empty     causal, with some rows given ke < 0 or ke <= ks.
    past_end  windows running past N, starts past N, and starts below 0.
    cp        two halves of a context-parallel split: the first M/2 rows
              are early positions, the rest late ones, of one request.
    """
    i = np.arange(m, dtype=np.int64)
    if mode == "causal":
        ks = np.zeros(m, np.int64)
        ke = n - m + i + 1
    elif mode in ("multi_req", "config3"):
        if mode == "config3":
            sizes = [m // requests] * requests
        else:
            cuts = np.sort(rng.choice(np.arange(1, m), requests - 1, replace=False))
            sizes = np.diff(np.concatenate([[0], cuts, [m]])).tolist()
        kv_per = n // requests
        ks = np.empty(m, np.int64)
        ke = np.empty(m, np.int64)
        r0 = 0
        for r, sz in enumerate(sizes):
            base = r * kv_per
            rows = np.arange(sz, dtype=np.int64)
            ks[r0: r0 + sz] = base
            ke[r0: r0 + sz] = base + kv_per - sz + rows + 1
            r0 += sz
    elif mode == "misaligned":
        off = 37
        ks = np.full(m, off, np.int64)
        ke = off + (n - off - m) + i + 1
    elif mode == "empty":
        ks = np.zeros(m, np.int64)
        ke = n - m + i + 1
        sel = rng.choice(m, max(1, m // 4), replace=False)
        half = sel[: len(sel) // 2]
        rest = sel[len(sel) // 2:]
        ke[half] = -rng.integers(1, 100, size=len(half))
        ks[rest] = ke[rest] + rng.integers(0, 50, size=len(rest))
    elif mode == "past_end":
        ks = rng.integers(0, n, size=m).astype(np.int64)
        ke = ks + rng.integers(1, n, size=m)
        sel = rng.choice(m, max(2, m // 4), replace=False)
        far, neg = sel[: len(sel) // 2], sel[len(sel) // 2:]
        ks[far] = n + rng.integers(0, 300, size=len(far))
        ke[far] = ks[far] + 50
        ks[neg] = -rng.integers(1, 200, size=len(neg))  # starts before 0
    elif mode == "cp":
        half = m // 2
        ks = np.zeros(m, np.int64)
        ke = np.empty(m, np.int64)
        ke[:half] = np.arange(half) + 1
        ke[half:] = n - (m - half) + np.arange(m - half) + 1
    else:
        raise ValueError(mode)
    return ks.astype(np.int32), ke.astype(np.int32)


def prefill_case(m, n, heads, dim=128, mode="causal", seed=0, requests=4,
                 name=""):
    rng = np.random.default_rng(seed)
    ks, ke = prefill_windows(mode, m, n, rng, requests)
    q = _q_codes(rng, (m, heads, dim))
    k, s = _k_tokens(rng, n, dim)
    w = _weights(rng, m, heads)
    return PrefillCase(q=q, k=k, kv_scale=s, weights=w, ks=ks, ke=ke, name=name)


# The five benchmark configurations (seed = 1000 + index).
CONFIGS = {
    0: dict(kind="decode", batch=1, next_n=1, heads=32, max_model_len=1024,
            block_size=64, context_lens=[1024],
            desc="decode B1 next_n1 H32 ctx1024 blk64"),
    1: dict(kind="decode", batch=16, next_n=2, heads=32, max_model_len=8192,
            block_size=64, var_ratio=0.3,
            desc="decode B16 next_n2 H32 mml8192 ragged(0.3) blk64"),
    2: dict(kind="decode", batch=16, next_n=6, heads=32, max_model_len=1048576,
            block_size=64, context_lens=[131072] * 16,
            desc="decode MTP-verify B16 next_n6 H32 ctx131072 mml1048576 blk64"),
    3: dict(kind="prefill", m=4096, n=32768, heads=32, mode="config3",
            requests=4, desc="prefill M4096 N32768 H32 4x1024 causal rows"),
    # the prefill page's other real chunk shapes (one causal request per chunk)
    5: dict(kind="prefill", m=2048, n=65536, heads=32, mode="causal", requests=1,
            desc="prefill M2048 N65536 H32 one causal request"),
    6: dict(kind="prefill", m=1024, n=131072, heads=32, mode="causal", requests=1,
            desc="prefill M1024 N131072 H32 one causal request"),
    4: dict(kind="decode", batch=64, next_n=4, heads=64, max_model_len=32768,
            block_size=1, var_ratio=0.3,
            desc="decode B64 next_n4 H64 mml32768 ragged(0.3) blk1"),
}


def make_config(idx: int, next_n: int | None = None):
    """Build benchmark configuration `idx` (optionally overriding next_n)."""
    c = dict(CONFIGS[idx])
    kind = c.pop("kind")
    desc = c.pop("desc")
    seed = 1000 + idx
    if kind == "decode":
        if next_n is not None:
            c["next_n"] = next_n
        return decode_case(seed=seed, name=desc, **c)
    return prefill_case(seed=seed, name=desc, **c)


@dataclasses.dataclass
class PagedPrefillCase:
    q: np.ndarray             # [M, H, D] u8
    kv_cache: np.ndarray      # [num_blocks, block_size*(D+4)] u8
    block_tables: np.ndarray  # [R, max_blocks] i32
    cu_seq_lens: np.ndarray   # [R + 1] i32
    weights: np.ndarray       # [M, H] f32
    ks: np.ndarray            # [M] i32
    ke: np.ndarray            # [M] i32
    block_size: int
    name: str = ""

    @property
    def rows(self):
        return self.q.shape[0]

    @property
    def cols(self):
        return int(self.cu_seq_lens[-1])

    @property
    def heads(self):
        return self.q.shape[1]


def paged_prefill_case(seq_lens, rows_per_req, heads, block_size=64, dim=128, seed=0, poison=False,
                       extra_blocks=0, name=""):
    """Requests with K lengths seq_lens in a permuted paged cache (as in
    decode_case); request r contributes rows_per_req[r] query rows, the last
    positions of the request (causal chunk): row i of request r has window
    [cu[r], cu[r] + len_r - rows_r + i + 1) in the gathered columns."""
    seq = np.asarray(seq_lens, dtype=np.int64)
    rows = np.asarray(rows_per_req, dtype=np.int64)
    mml = max(int(seq.max()) if seq.size else 1, 1)
    base = decode_case(seq.size, 1, heads, dim=dim, max_model_len=mml, block_size=block_size,
                       context_lens=seq, seed=seed, poison=poison, extra_blocks=extra_blocks)
    rng = np.random.default_rng(seed + 7)
    cu = np.concatenate([[0], np.cumsum(seq)]).astype(np.int32)
    ks, ke = [], []
    for r in range(seq.size):
        for i in range(int(rows[r])):
            ks.append(cu[r])
            ke.append(cu[r] + seq[r] - rows[r] + i + 1)
    m = len(ks)
    q = _q_codes(rng, (m, heads, dim))
    w = _weights(rng, m, heads)
    return PagedPrefillCase(q=q, kv_cache=base.kv_cache, block_tables=base.block_tables, cu_seq_lens=cu,
                            weights=w, ks=np.asarray(ks, np.int32), ke=np.asarray(ke, np.int32),
                            block_size=block_size, name=name)
