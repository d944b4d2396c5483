"""CPU oracle for the FP8 indexer logits -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / ``--impl reference`` legs may import this package.  The
product library never does, and this package imports nothing from it.

The arithmetic lives in ``fp8idx_oracle.c`` (plain C, fp64, OpenMP); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8idx_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle C source into a shared object (gcc -O2, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", *extra_flags, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


class PagedArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("kv_cache", ctypes.c_void_p),
        ("weights", ctypes.c_void_p), ("context_lens", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p), ("num_blocks", ctypes.c_int64),
        ("block_size", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
        ("batch", ctypes.c_int32), ("next_n", ctypes.c_int32),
        ("heads", ctypes.c_int32), ("dim", ctypes.c_int32),
        ("max_model_len", ctypes.c_int32),
    ]


class PrefillArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p),
        ("kv_scale", ctypes.c_void_p), ("weights", ctypes.c_void_p),
        ("ks", ctypes.c_void_p), ("ke", ctypes.c_void_p),
        ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
        ("heads", ctypes.c_int32), ("dim", ctypes.c_int32),
    ]


def _bind(lib):
    P = ctypes.c_void_p
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    for name, argt in (("oracle_paged_mqa_logits", PagedArgs),
                       ("oracle_mqa_logits", PrefillArgs)):
        fn = getattr(lib, name)
        fn.argtypes = [ctypes.POINTER(argt), ctypes.c_int64, ctypes.c_int64, P]
        fn.restype = ctypes.c_int
        fn_at = getattr(lib, name + "_at")
        fn_at.argtypes = [ctypes.POINTER(argt), ctypes.c_int64, P, P, P]
        fn_at.restype = ctypes.c_int
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` loads a variant."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(_LIB_PATH)
                     or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
            if stale:
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """numpy-facing wrapper around one loaded oracle library."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def e4m3_to_double(self, code: int) -> float:
        return float(self.lib.oracle_e4m3_to_double(code))

    # -- decode ---------------------------------------------------------------
    def _paged(self, q, kv_cache, weights, context_lens, block_tables,
               block_size, max_model_len):
        q = _c(q, np.uint8)
        kv = _c(kv_cache, np.uint8)
        w = _c(weights, np.float32)
        cl = _c(context_lens, np.int32)
        bt = _c(block_tables, np.int32)
        batch, next_n, heads, dim = q.shape
        assert w.shape == (batch * next_n, heads)
        assert bt.shape[0] == batch and cl.shape == (batch,)
        assert kv.shape[1] == block_size * (dim + 4)
        args = PagedArgs(q.ctypes.data, kv.ctypes.data, w.ctypes.data,
                         cl.ctypes.data, bt.ctypes.data, kv.shape[0],
                         block_size, bt.shape[1], batch, next_n, heads, dim,
                         max_model_len)
        keep = (q, kv, w, cl, bt)
        return args, keep, batch * next_n

    def paged_mqa_logits(self, q, kv_cache, weights, context_lens, block_tables,
                         block_size, max_model_len, rows=None):
        """Dense decode logits [rows, max_model_len] (float64, -inf outside)."""
        args, keep, nrows = self._paged(q, kv_cache, weights, context_lens,
                                        block_tables, block_size, max_model_len)
        r0, r1 = (0, nrows) if rows is None else rows
        out = np.empty((r1 - r0, max_model_len), np.float64)
        rc = self.lib.oracle_paged_mqa_logits(ctypes.byref(args), r0, r1,
                                              out.ctypes.data)
        if rc != 0:
            raise ValueError("oracle: block id or context length out of range")
        del keep
        return out

    def paged_mqa_logits_at(self, q, kv_cache, weights, context_lens,
                            block_tables, block_size, max_model_len, rows, cols):
        args, keep, _ = self._paged(q, kv_cache, weights, context_lens,
                                    block_tables, block_size, max_model_len)
        rows = _c(rows, np.int64)
        cols = _c(cols, np.int64)
        vals = np.empty(rows.shape, np.float64)
        rc = self.lib.oracle_paged_mqa_logits_at(
            ctypes.byref(args), rows.size, rows.ctypes.data, cols.ctypes.data,
            vals.ctypes.data)
        if rc != 0:
            raise ValueError("oracle: block id or context length out of range")
        del keep
        return vals

    # -- prefill --------------------------------------------------------------
    def _prefill(self, q, k, kv_scale, weights, ks, ke):
        q = _c(q, np.uint8)
        k = _c(k, np.uint8)
        s = _c(kv_scale, np.float32)
        w = _c(weights, np.float32)
        ks = _c(ks, np.int32)
        ke = _c(ke, np.int32)
        m, heads, dim = q.shape
        n = k.shape[0]
        assert k.shape == (n, dim) and s.shape == (n,)
        assert w.shape == (m, heads) and ks.shape == (m,) and ke.shape == (m,)
        args = PrefillArgs(q.ctypes.data, k.ctypes.data, s.ctypes.data,
                           w.ctypes.data, ks.ctypes.data, ke.ctypes.data, m, n,
                           heads, dim)
        return args, (q, k, s, w, ks, ke), m, n

    def mqa_logits(self, q, k, kv_scale, weights, ks, ke, rows=None):
        """Dense prefill logits [rows, N] (float64, -inf outside windows)."""
        args, keep, m, n = self._prefill(q, k, kv_scale, weights, ks, ke)
        r0, r1 = (0, m) if rows is None else rows
        out = np.empty((r1 - r0, n), np.float64)
        self.lib.oracle_mqa_logits(ctypes.byref(args), r0, r1, out.ctypes.data)
        del keep
        return out

    def mqa_logits_at(self, q, k, kv_scale, weights, ks, ke, rows, cols):
        args, keep, _, _ = self._prefill(q, k, kv_scale, weights, ks, ke)
        rows = _c(rows, np.int64)
        cols = _c(cols, np.int64)
        vals = np.empty(rows.shape, np.float64)
        self.lib.oracle_mqa_logits_at(ctypes.byref(args), rows.size,
                                      rows.ctypes.data, cols.ctypes.data,
                                      vals.ctypes.data)
        del keep
        return vals


def gather_paged_k(kv_cache, block_tables, cu_seq_lens, block_size: int, dim: int = 128):
    """The caller's gather the prefill page describes (aiter PR 5046,
    Motivation: K gathered out of the paged cache into a contiguous [N, 128]
    buffer with a separate [N] f32 scale): request r's tokens t < its length
    cu[r+1] - cu[r] come from slot t % block_size of block
    block_tables[r][t // block_size]; a block holds block_size rows of `dim`
    e4m3 bytes followed by block_size f32 scales.  Plain numpy indexing."""
    kv = np.asarray(kv_cache, dtype=np.uint8)
    cu = np.asarray(cu_seq_lens, dtype=np.int64)
    n = int(cu[-1])
    k = np.zeros((n, dim), np.uint8)
    s = np.zeros((n,), np.float32)
    for r in range(cu.size - 1):
        for t in range(int(cu[r + 1] - cu[r])):
            blk = int(block_tables[r][t // block_size])
            slot = t % block_size
            page = kv[blk]
            k[cu[r] + t] = page[slot * dim:(slot + 1) * dim]
            s[cu[r] + t] = page[block_size * dim + 4 * slot: block_size * dim + 4 * slot + 4].view(np.float32)[0]
    return k, s
