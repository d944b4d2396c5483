"""GPU parity of fp8_mqa_logits (prefill) against the CPU oracle.

The output is NaN-poisoned before every call; prefill writes every element
(-inf outside the windows), so any position left unwritten fails the -inf
mask check.  The window modes are the ones the prefill pages grade: causal,
multi-request packing, a misaligned start, empty rows, windows past the end
(and before the start), and a context-parallel split.
"""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_rows_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8idx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_fp8_gb300 as m
    m.library()
    return m


def run_prefill(fp8idx, case, options=None, clean_logits=True):
    d = to_device(case)
    out = torch.full((case.rows, case.cols), float("nan"), dtype=torch.float32, device="cuda")
    fp8idx.fp8_mqa_logits(d["q"], d["k"], d["kv_scale"], d["weights"], d["ks"], d["ke"], out, options=options,
                          clean_logits=clean_logits)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def oracle_prefill(o, case, rows=None):
    return o.mqa_logits(case.q, case.k, case.kv_scale, case.weights, case.ks, case.ke, rows=rows)


MODES = ["causal", "multi_req", "misaligned", "empty", "past_end", "cp"]


@pytest.mark.parametrize("heads", [32, 64, 128])
@pytest.mark.parametrize("mode", MODES)
def test_prefill_window_modes(fp8idx, oracle_impl, mode, heads):
    # M not a multiple of the row block, N not a multiple of the 128-token tile
    case = workloads.prefill_case(45, 700, heads, mode=mode, seed=100 + MODES.index(mode))
    gpu = run_prefill(fp8idx, case)
    assert_rows_close(gpu, oracle_prefill(oracle_impl, case), what=f"{mode}/h{heads}")


@pytest.mark.parametrize("heads", [32, 64, 128])
@pytest.mark.parametrize("mode", MODES)
def test_prefill_head_dim_64(fp8idx, oracle_impl, mode, heads):
    """head_dim 64 (64-byte rows in the 64-byte swizzle, two K=32 MMAs per
    tile), the other head size of the pages' prefill sweep."""
    case = workloads.prefill_case(45, 700, heads, dim=64, mode=mode, seed=300 + MODES.index(mode))
    assert_rows_close(run_prefill(fp8idx, case), oracle_prefill(oracle_impl, case), what=f"d64 {mode}/h{heads}")


@pytest.mark.parametrize("opts", [dict(split_n=1), dict(block_m=3), dict(stages=2)], ids=["split1", "bm3", "st2"])
def test_prefill_head_dim_64_overrides_and_no_clean(fp8idx, oracle_impl, opts):
    case = workloads.prefill_case(70, 1300, 32, dim=64, mode="multi_req", seed=31)
    ref = oracle_prefill(oracle_impl, case)
    assert_rows_close(run_prefill(fp8idx, case, options=fp8idx.Options(**opts)), ref, what=f"d64 {opts}")
    gpu = run_prefill(fp8idx, case, options=fp8idx.Options(**opts), clean_logits=False)
    assert_rows_close(gpu, ref, written=np.isfinite(ref), what=f"d64 no-clean {opts}")


@pytest.mark.parametrize("heads", [32, 128])
@pytest.mark.parametrize("mode", MODES)
def test_prefill_no_clean_logits(fp8idx, oracle_impl, mode, heads):
    """clean_logits=False: exactly the windows are written (the NaN poison
    must survive everywhere else, including past_end windows that start
    beyond N, which the pages report as the out-of-bounds case)."""
    case = workloads.prefill_case(45, 701, heads, mode=mode, seed=200 + MODES.index(mode))
    gpu = run_prefill(fp8idx, case, clean_logits=False)
    ref = oracle_prefill(oracle_impl, case)
    assert_rows_close(gpu, ref, written=np.isfinite(ref), what=f"no-clean {mode}/h{heads}")


@pytest.mark.parametrize("shape", [(1, 1), (3, 128), (8, 129), (17, 256), (64, 1000), (200, 520)])
def test_prefill_shapes(fp8idx, oracle_impl, shape):
    m, n = shape
    case = workloads.prefill_case(m, n, 32, mode="causal" if m <= n else "past_end", seed=m * 7 + n)
    gpu = run_prefill(fp8idx, case)
    assert_rows_close(gpu, oracle_prefill(oracle_impl, case), what=str(shape))


@pytest.mark.parametrize("opts", [dict(split_n=1), dict(split_n=5), dict(reverse_rows=0), dict(reverse_rows=1),
                                  dict(block_m=3), dict(stages=2), dict(block_m=1, split_n=2)],
                         ids=["split1", "split5", "natural", "reverse", "block_m3", "stages2", "block_m1"])
def test_prefill_planner_overrides(fp8idx, oracle_impl, opts):
    case = workloads.prefill_case(70, 900, 32, mode="multi_req", seed=9)
    gpu = run_prefill(fp8idx, case, options=fp8idx.Options(**opts))
    assert_rows_close(gpu, oracle_prefill(oracle_impl, case), what=str(opts))


@pytest.mark.slow
def test_prefill_config3_full_size(fp8idx, oracle_impl):
    """Full 4096 x 32768 run compared with the oracle element by element:
    every row (oracle streamed in chunks of 256 rows), the exact -inf mask,
    and each finite logit against its own row's oracle maximum."""
    case = workloads.make_config(3)
    gpu = run_prefill(fp8idx, case)
    for r0 in range(0, case.rows, 256):
        r1 = min(case.rows, r0 + 256)
        assert_rows_close(gpu[r0:r1], oracle_prefill(oracle_impl, case, rows=(r0, r1)), what=f"rows {r0}..{r1}")


@pytest.mark.slow
@pytest.mark.parametrize("m,n", [(2048, 65536), (1024, 131072)], ids=["2048x65536", "1024x131072"])
def test_prefill_real_chunk_shapes(fp8idx, oracle_impl, m, n):
    """The pages' other real chunk shapes (one causal request per chunk).
    Each holds about 1.3e8 window logits, several minutes of the fp64 oracle,
    so: the exact -inf mask of every element, full oracle rows at both ends
    and in the middle, and 256 random in-window elements of EVERY row, each
    judged against that row's largest sampled oracle magnitude (a lower bound
    of the row maximum, so the bar applied is at least as strict as the
    per-row one)."""
    case = workloads.prefill_case(m, n, 32, mode="causal", seed=m + n)
    gpu = run_prefill(fp8idx, case)
    cols = np.arange(n)[None, :]
    for r0 in range(0, m, 128):
        lo = np.maximum(case.ks[r0:r0 + 128].astype(np.int64), 0)[:, None]
        hi = np.minimum(case.ke[r0:r0 + 128].astype(np.int64), n)[:, None]
        inside = (cols >= lo) & (cols < hi)
        assert np.array_equal(np.isneginf(gpu[r0:r0 + 128]), ~inside), f"rows {r0}..: -inf mask"
    for r in (0, m // 2, m - 1):
        ref = oracle_prefill(oracle_impl, case, rows=(r, r + 1))
        assert_rows_close(gpu[r:r + 1], ref, what=f"row {r}")
    per_row = 256
    rng = np.random.default_rng(2)
    rows = np.repeat(np.arange(m, dtype=np.int64), per_row)
    lo = np.maximum(case.ks[rows].astype(np.int64), 0)
    hi = np.minimum(case.ke[rows].astype(np.int64), n)
    assert (hi > lo).all()
    cols_s = lo + (rng.random(rows.size) * (hi - lo)).astype(np.int64)
    ref = oracle_impl.mqa_logits_at(case.q, case.k, case.kv_scale, case.weights, case.ks, case.ke, rows, cols_s)
    rowmax = np.abs(ref).reshape(m, per_row).max(axis=1)
    tol = 1e-3 * np.repeat(rowmax, per_row) + 1e-5
    err = np.abs(gpu[rows, cols_s].astype(np.float64) - ref)
    bad = err > tol
    assert not bad.any(), f"{int(bad.sum())} sampled logits out of tolerance, max err {err.max()}"


@pytest.mark.parametrize("cols,pitch", [(701, 704), (701, 705), (130, 132), (64, 256)],
                         ids=["aligned-pitch", "odd-pitch", "tail2", "wide-pitch"])
def test_prefill_strided_out(fp8idx, oracle_impl, cols, pitch):
    """out is a column slice of a wider NaN buffer: the -inf fill (TMA stores
    clipped at column N when the pitch is a multiple of 4 floats, thread
    stores otherwise) must write [0, N) of every row and nothing past it."""
    case = workloads.prefill_case(37, cols, 32, mode="multi_req", seed=cols + pitch)
    d = to_device(case)
    buf = torch.full((case.rows, pitch), float("nan"), dtype=torch.float32, device="cuda")
    out = buf[:, :cols]
    fp8idx.fp8_mqa_logits(d["q"], d["k"], d["kv_scale"], d["weights"], d["ks"], d["ke"], out)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    assert np.isnan(host[:, cols:]).all(), "columns past N were written"
    assert_rows_close(host[:, :cols], oracle_prefill(oracle_impl, case), what=f"N={cols} pitch={pitch}")


def test_prefill_graph_capture_replay(fp8idx, oracle_impl):
    case = workloads.prefill_case(40, 600, 32, mode="multi_req", seed=41)
    d = to_device(case)
    out = torch.full((40, 600), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fp8idx.fp8_mqa_logits(d["q"], d["k"], d["kv_scale"], d["weights"], d["ks"], d["ke"], out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fp8idx.fp8_mqa_logits(d["q"], d["k"], d["kv_scale"], d["weights"], d["ks"], d["ke"], out, stream=s)
    case2 = workloads.prefill_case(40, 600, 32, mode="multi_req", seed=42)
    for key in ("q", "k", "kv_scale", "weights", "ks", "ke"):
        d[key].copy_(torch.from_numpy(getattr(case2, key)))
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert_rows_close(out.cpu().numpy(), oracle_prefill(oracle_impl, case2), what="graph replay")


def test_prefill_empty_and_errors(fp8idx):
    case = workloads.prefill_case(4, 64, 32, seed=5)
    d = to_device(case)
    empty = torch.empty((0, 64), device="cuda")
    fp8idx.fp8_mqa_logits(d["q"][:0], d["k"], d["kv_scale"], d["weights"][:0], d["ks"][:0], d["ke"][:0], empty)
    out = torch.full((4, 64), float("nan"), device="cuda")
    with pytest.raises(fp8idx.Fp8IdxError) as e:
        fp8idx.fp8_mqa_logits(d["q"], d["k"], d["kv_scale"], d["weights"], d["ks"], d["ke"][:3], out)
    assert e.value.status == fp8idx.FP8IDX_ERR_INVALID
    torch.cuda.synchronize()
    assert fp8idx.device_status() == fp8idx.FP8IDX_OK
