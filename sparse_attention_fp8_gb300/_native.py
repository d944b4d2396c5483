"""ctypes binding of libfp8idx (argument marshalling only)."""
from __future__ import annotations

import ctypes
import dataclasses
import os
import re
import struct
import threading

from . import _build

FP8IDX_OK = 0
FP8IDX_ERR_INVALID = 1
FP8IDX_ERR_UNSUPPORTED = 2
FP8IDX_ERR_CUDA = 3
FP8IDX_ERR_TIMEOUT = 4
_STATUS_NAMES = {0: "OK", 1: "INVALID", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT"}

_U8, _F32, _I32 = 0, 1, 2


class Fp8IdxError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"fp8idx {_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _Tensor(ctypes.Structure):
    """fp8idx_tensor as a ctypes structure (tests build descriptors by hand)."""
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


# fp8idx_tensor packed in one call (data, dtype, ndim, shape[4], stride[4]):
# the descriptors of a call are bytes objects handed to the library as
# pointers, which costs a third of filling ctypes structures field by field.
_TENSOR_PACK = struct.Struct("=qii4q4q")
assert _TENSOR_PACK.size == ctypes.sizeof(_Tensor)
_PAD = (0, 0, 0, 0)
_dtype_codes = None


class _Options(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int32), ("stages", ctypes.c_int32), ("split_n", ctypes.c_int32),
                ("reverse_rows", ctypes.c_int32), ("block_m", ctypes.c_int32), ("clean_logits", ctypes.c_int32)]


class _Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("grid", "threads", "smem_bytes", "stages", "tile_n", "block_m",
                                               "split_n", "reverse_rows", "tmem_cols", "gather")]


@dataclasses.dataclass
class Options:
    """Tunables; 0 (or -1 for reverse_rows) = host heuristic.  clean_logits:
    0/1 = write -inf outside the prefill windows, -1 = leave them untouched."""
    num_ctas: int = 0
    stages: int = 0
    split_n: int = 0
    reverse_rows: int = -1
    block_m: int = 0
    clean_logits: int = 0

    def _c(self):
        return _Options(self.num_ctas, self.stages, self.split_n, self.reverse_rows, self.block_m,
                        self.clean_logits)


@dataclasses.dataclass
class Plan:
    grid: int
    threads: int
    smem_bytes: int
    stages: int
    tile_n: int
    block_m: int
    split_n: int
    reverse_rows: int
    tmem_cols: int
    gather: int


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def library():
    """The loaded libfp8idx; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise ImportError(f"libfp8idx.so not built ({path}); run __graft_entry__.build() "
                                  "or python sparse_attention_fp8_gb300/_build.py")
            lib = ctypes.CDLL(path)
            P = ctypes.POINTER
            T = ctypes.c_void_p  # const fp8idx_tensor*: a packed descriptor, or byref(_Tensor)
            V = ctypes.c_void_p
            lib.fp8_paged_mqa_logits.argtypes = [T, T, T, T, T, ctypes.c_int32, T, V]
            lib.fp8_paged_mqa_logits_ex.argtypes = [T, T, T, T, T, ctypes.c_int32, T, P(_Options), V]
            lib.fp8_mqa_logits.argtypes = [T, T, T, T, T, T, T, V]
            lib.fp8_mqa_logits_ex.argtypes = [T, T, T, T, T, T, T, P(_Options), V]
            lib.fp8_mqa_logits_paged.argtypes = [T, T, T, T, T, T, T, T, P(_Options), V]
            lib.fp8_paged_topk.argtypes = [T, T, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, T, V]
            lib.fp8_mqa_topk.argtypes = [T, T, T, ctypes.c_int32, T, V]
            lib.fp8_paged_topk_ex.argtypes = [T, T, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, T, P(_Options), V]
            lib.fp8_mqa_topk_ex.argtypes = [T, T, T, ctypes.c_int32, T, P(_Options), V]
            lib.fp8_paged_mqa_topk.argtypes = [T, T, T, T, T, ctypes.c_int32, ctypes.c_int32, T, V,
                                               ctypes.c_size_t, P(_Options), V]
            lib.fp8_paged_mqa_topk.restype = ctypes.c_int
            lib.fp8idx_paged_mqa_topk_workspace.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                            ctypes.c_int32]
            lib.fp8idx_paged_mqa_topk_workspace.restype = ctypes.c_size_t
            for f in ("fp8_paged_mqa_logits", "fp8_paged_mqa_logits_ex", "fp8_mqa_logits", "fp8_mqa_logits_ex",
                      "fp8_mqa_logits_paged", "fp8_paged_topk", "fp8_mqa_topk", "fp8_paged_topk_ex",
                      "fp8_mqa_topk_ex"):
                getattr(lib, f).restype = ctypes.c_int
            lib.fp8idx_paged_is_supported.argtypes = [ctypes.c_int32] * 4
            lib.fp8idx_paged_is_supported.restype = ctypes.c_int
            lib.fp8idx_prefill_is_supported.argtypes = [ctypes.c_int32] * 2
            lib.fp8idx_prefill_is_supported.restype = ctypes.c_int
            lib.fp8idx_is_supported.argtypes = [ctypes.c_int32] * 4
            lib.fp8idx_is_supported.restype = ctypes.c_int
            lib.fp8idx_plan_paged.argtypes = [ctypes.c_int32] * 7 + [P(_Options), P(_Plan)]
            lib.fp8idx_plan_paged.restype = ctypes.c_int
            lib.fp8idx_plan_prefill.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                ctypes.c_int32, P(_Options), P(_Plan)]
            lib.fp8idx_plan_prefill.restype = ctypes.c_int
            lib.fp8idx_last_error.restype = ctypes.c_char_p
            lib.fp8idx_device_status.argtypes = [ctypes.c_int32]
            lib.fp8idx_device_status.restype = ctypes.c_int
            lib.fp8idx_host_mapped_pointer.argtypes = [V, P(ctypes.c_void_p)]
            lib.fp8idx_host_mapped_pointer.restype = ctypes.c_int
            lib.fp8idx_version.restype = ctypes.c_int32
            lib.fp8idx_watchdog_selftest.argtypes = [ctypes.c_int32, ctypes.c_void_p]
            lib.fp8idx_watchdog_selftest.restype = ctypes.c_int
            _lib = lib
    return _lib


def header_functions() -> list[str]:
    """Names of the functions declared in include/fp8idx.h."""
    path = os.path.join(_build.ROOT, "include", "fp8idx.h")
    with open(path) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", src, flags=re.M)


def _check(status: int):
    if status != FP8IDX_OK:
        msg = library().fp8idx_last_error()
        raise Fp8IdxError(status, msg.decode() if msg else "")


def _host_mapped(t) -> int:
    """Device address of a pinned host tensor (an output the kernel writes
    straight into host memory)."""
    if not t.is_pinned():
        raise ValueError("a host output must be a pinned (page-locked) tensor")
    dev = ctypes.c_void_p()
    _check(library().fp8idx_host_mapped_pointer(ctypes.c_void_p(t.data_ptr()), ctypes.byref(dev)))
    return dev.value


def _pack(t, ptr: int) -> bytes:
    """Packs tensor t's dtype, shape and strides with data address ptr into
    fp8idx_tensor bytes."""
    global _dtype_codes
    if _dtype_codes is None:
        import torch
        _dtype_codes = {torch.uint8: _U8, torch.float8_e4m3fn: _U8, torch.float32: _F32, torch.int32: _I32}
    dt = _dtype_codes.get(t.dtype)
    if dt is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    shape = t.shape
    n = len(shape)
    if n > 4:
        raise ValueError("at most 4 dimensions")
    return _TENSOR_PACK.pack(ptr, dt, n, *shape, *_PAD[n:], *t.stride(), *_PAD[n:])


def _desc(t, out: bool = False) -> bytes:
    """torch tensor -> packed fp8idx_tensor (no copy of the data; the tensor
    must outlive the call).  Inputs are CUDA tensors; an output (out=True) may
    also be a pinned host tensor, passed by its device mapping."""
    if t.is_cuda:
        return _pack(t, t.data_ptr())
    if not out:
        raise ValueError("inputs must be CUDA tensors")
    if t.numel() == 0:  # nothing is written: no address needed
        return _pack(t, 0)
    return _pack(t, _host_mapped(t))


def _stream(stream, like):
    import torch
    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)  # the current stream's handle, no object
        if raw is not None:
            return ctypes.c_void_p(raw(like.get_device()))
        return ctypes.c_void_p(torch.cuda.current_stream(like.device).cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def fp8_paged_mqa_logits(q_fp8, kv_cache, weights, context_lens, block_tables, max_model_len, out,
                         stream=None, options: Options | None = None):
    """Decode logits into ``out`` (only the causal windows are written).
    ``out`` may be a pinned host tensor: the kernel then writes the logits
    straight into host memory."""
    lib = library()
    args = [_desc(q_fp8), _desc(kv_cache), _desc(weights), _desc(context_lens), _desc(block_tables)]
    o = _desc(out, out=True)
    s = _stream(stream, q_fp8)
    if options is None:
        st = lib.fp8_paged_mqa_logits(*args, int(max_model_len), o, s)
    else:
        oc = options._c()
        st = lib.fp8_paged_mqa_logits_ex(*args, int(max_model_len), o, ctypes.byref(oc), s)
    _check(st)
    return out


def fp8_mqa_logits(q_fp8, k_fp8, kv_scale, weights, cu_seqlen_ks, cu_seqlen_ke, out, stream=None,
                   options: Options | None = None, clean_logits: bool = True):
    """Prefill logits into ``out``: every element written, -inf outside the
    windows (clean_logits=False: only the windows are written)."""
    if not clean_logits:
        options = dataclasses.replace(options or Options(), clean_logits=-1)
    lib = library()
    args = [_desc(q_fp8), _desc(k_fp8), _desc(kv_scale), _desc(weights), _desc(cu_seqlen_ks),
            _desc(cu_seqlen_ke)]
    o = _desc(out)
    s = _stream(stream, q_fp8)
    if options is None:
        st = lib.fp8_mqa_logits(*args, o, s)
    else:
        oc = options._c()
        st = lib.fp8_mqa_logits_ex(*args, o, ctypes.byref(oc), s)
    _check(st)
    return out


def fp8_mqa_logits_paged(q_fp8, kv_cache, block_tables, cu_seq_lens, weights, cu_seqlen_ks, cu_seqlen_ke, out,
                         stream=None, options: Options | None = None, clean_logits: bool = True):
    """Prefill logits with K read from the paged cache: column n of request r
    (cu_seq_lens[r] <= n < cu_seq_lens[r+1]) is its token n - cu_seq_lens[r]."""
    if not clean_logits:
        options = dataclasses.replace(options or Options(), clean_logits=-1)
    lib = library()
    args = [_desc(q_fp8), _desc(kv_cache), _desc(block_tables), _desc(cu_seq_lens), _desc(weights),
            _desc(cu_seqlen_ks), _desc(cu_seqlen_ke)]
    o = _desc(out)
    oc = options._c() if options is not None else None
    st = lib.fp8_mqa_logits_paged(*args, o, ctypes.byref(oc) if oc is not None else None, _stream(stream, q_fp8))
    _check(st)
    return out


def fp8_paged_topk(logits, context_lens, next_n, max_model_len, k, indices, stream=None, ctas_per_row: int = 0):
    """Decode top-k: indices [rows, k] of each row's k largest logits in its
    causal window (equal logits: lowest positions), listed by position, -1
    past the window.  ctas_per_row: 0 = heuristic, 1..8 = fixed (the result
    does not depend on it)."""
    lib = library()
    lg, cl, ix = _desc(logits), _desc(context_lens), _desc(indices, out=True)
    oc = Options(num_ctas=int(ctas_per_row))._c()
    _check(lib.fp8_paged_topk_ex(lg, cl, int(next_n), int(max_model_len), int(k), ix, ctypes.byref(oc),
                                 _stream(stream, logits)))
    return indices


def fp8_mqa_topk(logits, cu_seqlen_ks, cu_seqlen_ke, k, indices, stream=None, ctas_per_row: int = 0):
    """Prefill top-k over the windows [ks, ke) (same rule, order and padding)."""
    lib = library()
    lg, a, b, ix = _desc(logits), _desc(cu_seqlen_ks), _desc(cu_seqlen_ke), _desc(indices, out=True)
    oc = Options(num_ctas=int(ctas_per_row))._c()
    _check(lib.fp8_mqa_topk_ex(lg, a, b, int(k), ix, ctypes.byref(oc), _stream(stream, logits)))
    return indices


def paged_mqa_topk_workspace(batch, next_n, max_model_len, k) -> int:
    """Bytes of workspace fp8_paged_mqa_topk needs."""
    return int(library().fp8idx_paged_mqa_topk_workspace(int(batch), int(next_n), int(max_model_len), int(k)))


def fp8_paged_mqa_topk(q_fp8, kv_cache, weights, context_lens, block_tables, max_model_len, k, indices,
                       workspace=None, stream=None, options: Options | None = None):
    """Decode logits and their per-row top-k in one call (the logits of every
    row are never written): indices [batch*next_n, k] as fp8_paged_topk gives
    on the decode logits.  workspace: a uint8 CUDA tensor of at least
    paged_mqa_topk_workspace(...) bytes (allocated here if None)."""
    import torch
    lib = library()
    B, n = q_fp8.shape[0], q_fp8.shape[1]
    need = paged_mqa_topk_workspace(B, n, max_model_len, k)
    if workspace is None:
        workspace = torch.empty(need + 256, dtype=torch.uint8, device=q_fp8.device)
    base = workspace.data_ptr()
    off = (-base) % 256
    args = [_desc(q_fp8), _desc(kv_cache), _desc(weights), _desc(context_lens), _desc(block_tables)]
    ix = _desc(indices, out=True)
    oc = options._c() if options is not None else None
    st = lib.fp8_paged_mqa_topk(*args, int(max_model_len), int(k), ix,
                                ctypes.c_void_p(base + off), ctypes.c_size_t(workspace.numel() - off),
                                ctypes.byref(oc) if oc is not None else None, _stream(stream, q_fp8))
    _check(st)
    return indices


def paged_is_supported(heads, head_dim, block_size, next_n) -> bool:
    return bool(library().fp8idx_paged_is_supported(heads, head_dim, block_size, next_n))


def is_supported(heads, head_dim, kv_block_size, next_n) -> bool:
    """The decode gate (same as paged_is_supported)."""
    return bool(library().fp8idx_is_supported(heads, head_dim, kv_block_size, next_n))


def prefill_is_supported(heads, head_dim) -> bool:
    return bool(library().fp8idx_prefill_is_supported(heads, head_dim))


def _plan(pc: _Plan) -> Plan:
    return Plan(**{n: getattr(pc, n) for n, _ in _Plan._fields_})


def plan_paged(batch, next_n, heads, head_dim, block_size, max_model_len, num_sms=0,
               options: Options | None = None) -> Plan:
    pc = _Plan()
    oc = options._c() if options else None
    _check(library().fp8idx_plan_paged(batch, next_n, heads, head_dim, block_size, max_model_len, num_sms,
                                       ctypes.byref(oc) if oc else None, ctypes.byref(pc)))
    return _plan(pc)


def plan_prefill(rows, cols, heads, head_dim, num_sms=0, options: Options | None = None) -> Plan:
    pc = _Plan()
    oc = options._c() if options else None
    _check(library().fp8idx_plan_prefill(rows, cols, heads, head_dim, num_sms,
                                         ctypes.byref(oc) if oc else None, ctypes.byref(pc)))
    return _plan(pc)


def device_status(clear: bool = True) -> int:
    """FP8IDX_OK, or FP8IDX_ERR_TIMEOUT if an in-kernel wait ran out (synchronises)."""
    return int(library().fp8idx_device_status(1 if clear else 0))


def device_status_message() -> str:
    """The message of the last non-OK status (e.g. the watchdog's site bits)."""
    msg = library().fp8idx_last_error()
    return msg.decode() if msg else ""


def watchdog_selftest(limit_us: int = 5000, stream=None):
    """Enqueues the watchdog self-test: a bounded wait that nothing satisfies,
    given up after limit_us; afterwards device_status() reports a timeout."""
    import torch
    s = _stream(stream, torch.empty(0, device="cuda"))
    _check(library().fp8idx_watchdog_selftest(int(limit_us), s))


def version() -> int:
    return int(library().fp8idx_version())
