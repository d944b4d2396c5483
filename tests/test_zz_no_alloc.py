"""fp8_paged_mqa_topk_noalloc, the fused decode top-k for callers that
cannot allocate device memory (its scratch is a fixed static area inside
the library instead of a caller's workspace), called through the C ABI and
checked against fp8_paged_mqa_topk with a workspace: the indices must be
identical, on two calls in a row with different inputs (the second call
finds the first one's leftovers in the shared area).  Collected last, so a
run that stops at the first failure has run every other test first; it
also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from parity import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8idx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_fp8_gb300 as m
    m.library()
    return m


def noalloc_call(fp8idx, d, case, k, indices):
    from sparse_attention_fp8_gb300 import _native
    lib = fp8idx.library()
    fn = lib.fp8_paged_mqa_topk_noalloc
    T = ctypes.c_void_p  # const fp8idx_tensor*: the binding's packed descriptors
    fn.argtypes = [T, T, T, T, T, ctypes.c_int32, ctypes.c_int32, T, ctypes.POINTER(_native._Options),
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    descs = [_native._desc(d[key]) for key in ("q", "kv_cache", "weights", "context_lens", "block_tables")]
    ix = _native._desc(indices)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(*descs, case.max_model_len, k, ix, None, stream)


def with_workspace(fp8idx, d, case, k):
    out = torch.full((case.batch * case.next_n, k), -7, dtype=torch.int32, device="cuda")
    fp8idx.fp8_paged_mqa_topk(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                              case.max_model_len, k, out)
    return out


def test_noalloc_matches_workspace_entry_point_twice(fp8idx):
    cases = [
        (workloads.decode_case(4, 2, 32, max_model_len=20000, block_size=64, var_ratio=0.4, seed=61, poison=True,
                               extra_blocks=2), 512),
        (workloads.decode_case(3, 3, 64, max_model_len=9000, block_size=16, context_lens=[9000, 2500, 40], seed=62,
                               poison=True, extra_blocks=2), 2048),
    ]
    for i, (case, k) in enumerate(cases):
        d = to_device(case)
        got = torch.full((case.batch * case.next_n, k), -7, dtype=torch.int32, device="cuda")
        st = noalloc_call(fp8idx, d, case, k, got)
        assert st == fp8idx.FP8IDX_OK, fp8idx.library().fp8idx_last_error()
        want = with_workspace(fp8idx, d, case, k)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), want.cpu().numpy()), f"call {i + 1}"
    assert fp8idx.device_status() == fp8idx.FP8IDX_OK


def test_noalloc_rejects_shapes_beyond_its_scratch(fp8idx):
    """A shape whose scratch exceeds the static area is refused before any
    launch, with both sizes in the message."""
    case = workloads.decode_case(2, 4, 32, max_model_len=1 << 20, block_size=64, context_lens=[4096, 1000], seed=3)
    d = to_device(case)
    out = torch.empty((8, 64), dtype=torch.int32, device="cuda")
    st = noalloc_call(fp8idx, d, case, 64, out)
    assert st == fp8idx.FP8IDX_ERR_UNSUPPORTED
    msg = fp8idx.library().fp8idx_last_error().decode()
    assert "static scratch" in msg and "16777216" in msg, msg
