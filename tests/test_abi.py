"""The C-ABI library on the host (CPU only; nothing is launched).

Checks that libfp8idx.so loads, exports every function include/fp8idx.h
declares, and that the host-side logic (support gates, planner, argument
validation) behaves as documented.
"""
import ctypes

import pytest

import sparse_attention_fp8_gb300 as fp8idx
from sparse_attention_fp8_gb300 import _native


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_fp8_gb300 import _build
    _build.build()
    return fp8idx.library()


def test_exports_every_declared_function(lib):
    names = _native.header_functions()
    expected = {"fp8_paged_mqa_logits", "fp8_paged_mqa_logits_ex", "fp8_mqa_logits", "fp8_mqa_logits_ex",
                "fp8idx_paged_is_supported", "fp8idx_prefill_is_supported", "fp8idx_is_supported", "fp8idx_plan_paged",
                "fp8idx_plan_prefill", "fp8idx_last_error", "fp8idx_device_status", "fp8idx_version"}
    assert expected <= set(names), set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"


def test_version(lib):
    assert fp8idx.version() >= 100


def test_support_gates(lib):
    assert fp8idx.paged_is_supported(32, 128, 64, 6)
    assert fp8idx.paged_is_supported(32, 128, 1, 1)
    assert fp8idx.paged_is_supported(64, 128, 16, 4)
    assert not fp8idx.paged_is_supported(64, 128, 64, 5)   # next_n*heads > 256
    assert not fp8idx.paged_is_supported(32, 64, 64, 1)    # head_dim 64
    assert not fp8idx.paged_is_supported(16, 128, 64, 1)
    assert not fp8idx.paged_is_supported(32, 128, 8, 1)    # block size 8
    assert fp8idx.prefill_is_supported(32, 128) and fp8idx.prefill_is_supported(64, 128)
    assert fp8idx.prefill_is_supported(128, 128)
    assert fp8idx.prefill_is_supported(32, 64) and fp8idx.prefill_is_supported(128, 64)
    assert not fp8idx.prefill_is_supported(256, 128)
    assert not fp8idx.prefill_is_supported(32, 96)
    # the decode gate under its short name takes the same arguments and agrees
    for args in ((32, 128, 64, 6), (64, 128, 1, 4), (64, 128, 64, 5), (32, 64, 64, 1), (32, 128, 8, 1)):
        assert fp8idx.is_supported(*args) == fp8idx.paged_is_supported(*args), args


def test_planner_decode(lib):
    p = fp8idx.plan_paged(16, 6, 32, 128, 64, 1048576, num_sms=148)
    assert p.grid == 148 and p.tile_n == 192 and p.gather == 0
    assert p.smem_bytes <= 232448 and p.stages >= 4
    small = fp8idx.plan_paged(1, 1, 32, 128, 64, 1024, num_sms=148)
    assert small.grid == 4  # one CTA per 256-token item when there are fewer items than SMs
    g = fp8idx.plan_paged(64, 4, 64, 128, 1, 32768, num_sms=148)
    assert g.gather == 1 and g.tile_n == 256 and g.stages >= 6
    o = fp8idx.plan_paged(16, 6, 32, 128, 64, 1048576, num_sms=148, options=fp8idx.Options(num_ctas=7, stages=3))
    assert o.grid == 7 and o.stages == 3


def test_planner_prefill(lib):
    p = fp8idx.plan_prefill(4096, 32768, 32, 128, num_sms=148)
    assert p.block_m == 8 and p.tile_n == 256 and p.reverse_rows == 1
    assert p.grid == 148 and p.split_n >= 4  # persistent; >= 16 units per CTA
    assert p.smem_bytes <= 232448 and p.stages >= 4
    p64 = fp8idx.plan_prefill(1000, 1000, 64, 128, num_sms=148)
    assert p64.block_m == 4 and p64.reverse_rows == 0
    o = fp8idx.plan_prefill(4096, 32768, 32, 128, num_sms=148,
                            options=fp8idx.Options(split_n=3, reverse_rows=0, block_m=2))
    assert o.split_n == 3 and o.reverse_rows == 0 and o.tile_n == 64 and o.grid == 148
    small = fp8idx.plan_prefill(3, 100, 32, 128, num_sms=148)
    assert small.grid == 1 and small.split_n == 1  # one row block, one column tile
    with pytest.raises(fp8idx.Fp8IdxError) as e:
        fp8idx.plan_prefill(10, 10, 32, 128, num_sms=148, options=fp8idx.Options(block_m=9))
    assert e.value.status == fp8idx.FP8IDX_ERR_UNSUPPORTED


def _t(dtype, shape, ptr=0x1000):
    d = _native._Tensor()
    d.data = ptr
    d.dtype = dtype
    d.ndim = len(shape)
    st = 1
    for i in reversed(range(len(shape))):
        d.shape[i] = shape[i]
        d.stride[i] = st
        st *= shape[i]
    return d


def test_validation_rejects_before_touching_the_device(lib):
    """Malformed descriptors return INVALID from host checks (fake pointers,
    never dereferenced, no CUDA call reached)."""
    B, n, H, D = 2, 2, 32, 128
    q = _t(0, (B, n, H, D))
    kv = _t(0, (4, 64 * (D + 4)))
    w = _t(1, (B * n, H))
    cl = _t(2, (B,))
    bt = _t(2, (B, 2))
    out = _t(1, (B * n, 128))
    R = ctypes.byref
    st = lib.fp8_paged_mqa_logits(R(q), R(kv), R(_t(2, (B * n, H))), R(cl), R(bt), 128, R(out), None)
    assert st == fp8idx.FP8IDX_ERR_INVALID and b"weights" in lib.fp8idx_last_error()
    st = lib.fp8_paged_mqa_logits(None, R(kv), R(w), R(cl), R(bt), 128, R(out), None)
    assert st == fp8idx.FP8IDX_ERR_INVALID
    st = lib.fp8_paged_mqa_logits(R(q), R(_t(0, (4, 100))), R(w), R(cl), R(bt), 128, R(out), None)
    assert st == fp8idx.FP8IDX_ERR_INVALID  # cache row not block_size*(D+4)
    st = lib.fp8_paged_mqa_logits(R(q), R(kv), R(w), R(cl), R(bt), 129, R(out), None)
    assert st == fp8idx.FP8IDX_ERR_INVALID  # out narrower than max_model_len
    q16 = _t(0, (B, n, 16, D))
    st = lib.fp8_paged_mqa_logits(R(q16), R(kv), R(_t(1, (B * n, 16))), R(cl), R(bt), 128, R(out), None)
    assert st == fp8idx.FP8IDX_ERR_UNSUPPORTED
    qp = _t(0, (5, H, D))
    k = _t(0, (300, D))
    s = _t(1, (300,))
    wp = _t(1, (5, H))
    ks = _t(2, (5,))
    outp = _t(1, (5, 300))
    st = lib.fp8_mqa_logits(R(qp), R(k), R(s), R(wp), R(ks), R(_t(2, (4,))), R(outp), None)
    assert st == fp8idx.FP8IDX_ERR_INVALID
    st = lib.fp8_mqa_logits(R(qp), R(k), R(_t(1, (299,))), R(wp), R(ks), R(ks), R(outp), None)
    assert st == fp8idx.FP8IDX_ERR_INVALID


def test_descriptor_packing():
    """The binding packs each tensor into fp8idx_tensor bytes in one call:
    the same layout as the ctypes structure (pointer, dtype, ndim, shape[4],
    stride[4]), unused dimensions zero, strides in elements."""
    import torch
    t = torch.empty((3, 5, 7), dtype=torch.float32)[:, ::2, :]
    d = _native._Tensor.from_buffer_copy(_native._pack(t, 4096))
    assert d.data == 4096 and d.dtype == 1 and d.ndim == 3
    assert list(d.shape) == [3, 3, 7, 0] and list(d.stride) == [35, 14, 1, 0]
    u = torch.empty(16, dtype=torch.uint8)
    d = _native._Tensor.from_buffer_copy(_native._pack(u, u.data_ptr()))
    assert d.data == u.data_ptr()
    assert d.dtype == 0 and d.ndim == 1 and list(d.shape) == [16, 0, 0, 0] and list(d.stride) == [1, 0, 0, 0]
    with pytest.raises(TypeError):
        _native._pack(torch.empty(4, dtype=torch.float64), 0)
    with pytest.raises(ValueError):
        _native._pack(torch.empty((1, 1, 1, 1, 1), dtype=torch.float32), 0)
    # host tensors: never as inputs; as outputs only pinned (checked before any call)
    with pytest.raises(ValueError, match="inputs must be CUDA"):
        _native._desc(torch.empty(4, dtype=torch.float32))
    with pytest.raises(ValueError, match="pinned"):
        _native._desc(torch.empty(4, dtype=torch.float32), out=True)
    d = _native._Tensor.from_buffer_copy(_native._desc(torch.empty((0, 4), dtype=torch.int32), out=True))
    assert d.data is None and list(d.shape) == [0, 4, 0, 0]  # an empty host output needs no mapping


def test_host_mapped_pointer_arguments(lib):
    """The host-mapping query rejects null arguments before any CUDA call."""
    dev = ctypes.c_void_p()
    assert lib.fp8idx_host_mapped_pointer(None, ctypes.byref(dev)) == fp8idx.FP8IDX_ERR_INVALID
    assert lib.fp8idx_host_mapped_pointer(ctypes.c_void_p(4096), None) == fp8idx.FP8IDX_ERR_INVALID
    assert b"null" in lib.fp8idx_last_error()


def test_max_model_len_bound(lib):
    """Decode positions are kept in 32-bit registers: max_model_len above
    2^31 - 512 is UNSUPPORTED, reported by the host checks (fake pointers)."""
    B, n, H, D = 2, 2, 32, 128
    big = 0x7FFFFE01
    R = ctypes.byref
    st = lib.fp8_paged_mqa_logits(R(_t(0, (B, n, H, D))), R(_t(0, (4, 64 * (D + 4)))), R(_t(1, (B * n, H))),
                                  R(_t(2, (B,))), R(_t(2, (B, 2))), big, R(_t(1, (B * n, big))), None)
    assert st == fp8idx.FP8IDX_ERR_UNSUPPORTED and b"32 bits" in lib.fp8idx_last_error()
    # the fused decode top-k shares the decode set-up (and its bound)
    k = 8
    st = lib.fp8_paged_mqa_topk(R(_t(0, (B, n, H, D))), R(_t(0, (4, 64 * (D + 4)))), R(_t(1, (B * n, H))),
                                R(_t(2, (B,))), R(_t(2, (B, 2))), big, k, R(_t(2, (B * n, k))),
                                ctypes.c_void_p(0x100000), ctypes.c_size_t(1 << 40), None, None)
    assert st == fp8idx.FP8IDX_ERR_UNSUPPORTED and b"32 bits" in lib.fp8idx_last_error()


def test_misaligned_pointers_rejected(lib):
    """Operands read by TMA or bulk copies must be 16-byte aligned: an
    address 4 bytes off returns INVALID from the host checks, before any
    CUDA call (fake pointers, never dereferenced)."""
    R = ctypes.byref
    B, n, H, D = 2, 2, 32, 128
    good = dict(q=_t(0, (B, n, H, D)), kv=_t(0, (4, 64 * (D + 4))), w=_t(1, (B * n, H)), cl=_t(2, (B,)),
                bt=_t(2, (B, 2)), out=_t(1, (B * n, 128)))
    for name in ("q", "kv", "w"):
        a = dict(good)
        a[name] = _t(a[name].dtype, tuple(a[name].shape[:a[name].ndim]), ptr=0x1004)
        st = lib.fp8_paged_mqa_logits(R(a["q"]), R(a["kv"]), R(a["w"]), R(a["cl"]), R(a["bt"]), 128, R(a["out"]),
                                      None)
        assert st == fp8idx.FP8IDX_ERR_INVALID and b"aligned" in lib.fp8idx_last_error(), name
    M, N = 5, 300
    good = dict(q=_t(0, (M, H, D)), k=_t(0, (N, D)), s=_t(1, (N,)), w=_t(1, (M, H)), ks=_t(2, (M,)), ke=_t(2, (M,)),
                out=_t(1, (M, N)))
    for name in ("q", "k", "s", "w"):
        a = dict(good)
        a[name] = _t(a[name].dtype, tuple(a[name].shape[:a[name].ndim]), ptr=0x1004)
        st = lib.fp8_mqa_logits(R(a["q"]), R(a["k"]), R(a["s"]), R(a["w"]), R(a["ks"]), R(a["ke"]), R(a["out"]),
                                None)
        assert st == fp8idx.FP8IDX_ERR_INVALID and b"aligned" in lib.fp8idx_last_error(), name
    # paged prefill: a misaligned cache
    kv = _t(0, (8, 64 * (D + 4)), ptr=0x1008)
    bt = _t(2, (1, 8))
    cu = _t(2, (2,))
    st = lib.fp8_mqa_logits_paged(R(good["q"]), R(kv), R(bt), R(cu), R(good["w"]), R(good["ks"]), R(good["ke"]),
                                  R(good["out"]), None, None)
    assert st == fp8idx.FP8IDX_ERR_INVALID and b"aligned" in lib.fp8idx_last_error()


def test_watchdog_selftest_limit_checked_on_host(lib):
    """The self-test's wait limit is validated before any CUDA call."""
    for bad in (0, -5, 100001):
        assert lib.fp8idx_watchdog_selftest(bad, None) == fp8idx.FP8IDX_ERR_INVALID
        assert b"limit_us" in lib.fp8idx_last_error()


def test_fused_topk_workspace_size(lib):
    """The workspace size is a pure host function: zero for invalid
    arguments, growing with the rows and the width."""
    w = fp8idx.paged_mqa_topk_workspace(16, 6, 1048576, 2048)
    assert w >= 96 * 1048576 * 4  # a logits row per output row for the sample and the fallback
    assert fp8idx.paged_mqa_topk_workspace(16, 6, 1048576, 0) == 0
    assert fp8idx.paged_mqa_topk_workspace(16, 6, 1048576, 4096) == 0
    assert fp8idx.paged_mqa_topk_workspace(2, 1, 1000, 7) < fp8idx.paged_mqa_topk_workspace(4, 1, 1000, 7)
