"""GPU parity of the top-k consumers (fp8_paged_topk, fp8_mqa_topk) against
the numpy oracle (oracle/topk.py).  The result is unique by definition
(value descending, position ascending, -1 past the window), so indices must
match exactly.  Inputs cover the radix select's fast path (candidates in
shared memory) and its fallback (a top bin with more candidates than fit:
long runs of equal values), windows shorter than k, empty windows, -inf and
signed zeros, and logits produced by the library's own logits kernels.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import topk as T
from parity import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8idx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_fp8_gb300 as m
    m.library()
    return m


def gpu_mqa_topk(fp8idx, logits, ks, ke, k, ctas=0):
    lg = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    out = torch.full((logits.shape[0], k), -7, dtype=torch.int32, device="cuda")
    fp8idx.fp8_mqa_topk(lg, torch.from_numpy(ks).cuda(), torch.from_numpy(ke).cuda(), k, out, ctas_per_row=ctas)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def gpu_paged_topk(fp8idx, logits, context_lens, next_n, mml, k, ctas=0):
    lg = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    out = torch.full((logits.shape[0], k), -7, dtype=torch.int32, device="cuda")
    fp8idx.fp8_paged_topk(lg, torch.from_numpy(context_lens).cuda(), next_n, mml, k, out, ctas_per_row=ctas)
    torch.cuda.synchronize()
    return out.cpu().numpy()


MODES = ["causal", "multi_req", "misaligned", "empty", "past_end", "cp"]


@pytest.mark.parametrize("k", [1, 7, 512, 2048])
@pytest.mark.parametrize("mode", MODES)
def test_mqa_topk_window_modes(fp8idx, mode, k):
    rng = np.random.default_rng(MODES.index(mode) * 10 + k)
    m, n = 37, 5000
    ks, ke = workloads.prefill_windows(mode, m, n, rng, 4)
    logits = rng.normal(size=(m, n)).astype(np.float32)
    logits[:, ::13] = np.round(logits[:, ::13], 1)  # some exact ties
    want = T.topk_rows(logits, *T.prefill_windows(ks, ke, n), k)
    assert np.array_equal(gpu_mqa_topk(fp8idx, logits, ks, ke, k), want), f"{mode} k={k}"


@pytest.mark.parametrize("k", [512, 2048])
def test_mqa_topk_short_long_boundary(fp8idx, k):
    """Windows on both sides of the length where the selection moves from
    the whole window in shared memory (at most 8188 values: bulk copy into
    the key array, per-thread runs of up to 17 keys) to the sampled
    threshold and candidate compaction, starting at every offset modulo 4
    (the staged copy's 0-3 value lead-in)."""
    rng = np.random.default_rng(k)
    lens = [k + 1, 8183, 8187, 8188, 8189, 8192, 8193, 12000, 16384]
    m, n = len(lens) * 4, 20000
    ks = np.zeros(m, np.int32)
    ke = np.zeros(m, np.int32)
    for i, L in enumerate(lens):
        for off in range(4):
            s0 = int(rng.integers(0, n - L - 4)) // 4 * 4 + off
            ks[4 * i + off], ke[4 * i + off] = s0, s0 + L
    logits = rng.normal(size=(m, n)).astype(np.float32)
    logits[:, ::17] = np.round(logits[:, ::17], 1)  # some exact ties
    want = T.topk_rows(logits, *T.prefill_windows(ks, ke, n), k)
    assert np.array_equal(gpu_mqa_topk(fp8idx, logits, ks, ke, k), want), f"k={k}"


@pytest.mark.parametrize("levels", [1, 3, 50, 4000])
def test_mqa_topk_ties(fp8idx, levels):
    """Few distinct values: the top radix bin holds more candidates than
    shared memory (the fallback passes) and the tie rule decides."""
    rng = np.random.default_rng(levels)
    m, n = 6, 40000
    logits = rng.integers(0, levels, size=(m, n)).astype(np.float32) - levels / 2
    ks = np.array([0, 0, 100, 5000, 39000, 0], dtype=np.int32)
    ke = np.array([40000, 2047, 40000, 30000, 40000, 0], dtype=np.int32)
    for k in (1, 100, 2048):
        want = T.topk_rows(logits, *T.prefill_windows(ks, ke, n), k)
        assert np.array_equal(gpu_mqa_topk(fp8idx, logits, ks, ke, k), want), f"levels={levels} k={k}"


def test_mqa_topk_special_values(fp8idx):
    rng = np.random.default_rng(5)
    m, n = 8, 3000
    logits = rng.normal(size=(m, n)).astype(np.float32)
    logits[0, :] = 0.0
    logits[0, ::2] = -0.0                      # signed zeros compare equal
    logits[1, 100:2900] = -np.inf             # -inf inside the window
    logits[2, :] = np.float32(1e-40)          # subnormals
    logits[2, 7::9] = np.float32(-1e-40)
    logits[3, :] = -np.abs(logits[3, :])      # all negative
    logits[4, ::3] = np.inf
    ks = np.zeros(m, dtype=np.int32)
    ke = np.full(m, n, dtype=np.int32)
    for k in (1, 33, 2048):
        want = T.topk_rows(logits, *T.prefill_windows(ks, ke, n), k)
        assert np.array_equal(gpu_mqa_topk(fp8idx, logits, ks, ke, k), want), f"k={k}"


@pytest.mark.parametrize("shift,pad", [(1, 1), (2, 6), (0, 3)], ids=["unaligned-base", "shift2", "odd-stride"])
def test_mqa_topk_unaligned_rows(fp8idx, shift, pad):
    """Rows that do not start on 16 bytes (scalar loads) and windows with
    partial 4-value groups at both ends."""
    rng = np.random.default_rng(shift * 7 + pad)
    m, n = 21, 9000
    ks, ke = workloads.prefill_windows("past_end", m, n, rng, 4)
    buf = torch.from_numpy(rng.normal(size=(m, n + pad)).astype(np.float32)).cuda()
    lg = buf[:, shift:shift + n]
    want = T.topk_rows(lg.cpu().numpy(), *T.prefill_windows(ks, ke, n), 1000)
    out = torch.full((m, 1000), -7, dtype=torch.int32, device="cuda")
    fp8idx.fp8_mqa_topk(lg, torch.from_numpy(ks).cuda(), torch.from_numpy(ke).cuda(), 1000, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("ctas", [0, 1, 3, 8])
def test_paged_topk_ragged(fp8idx, ctas):
    rng = np.random.default_rng(11)
    batch, next_n, mml = 9, 3, 70000
    ctx = np.array([0, 1, 2, 3, 100, 2049, 2050, 69999, 70000], dtype=np.int32)
    logits = rng.normal(size=(batch * next_n, mml + 5)).astype(np.float32)  # wider than max_model_len
    for k in (1, 512, 2048):
        want = T.topk_rows(logits, *T.decode_windows(ctx, next_n, mml), k)
        assert np.array_equal(gpu_paged_topk(fp8idx, logits, ctx, next_n, mml, k, ctas), want), f"k={k}"


def test_topk_into_pinned_host_memory(fp8idx):
    """Pinned host index buffers: the kernels write the indices straight into
    host memory, the same as into device memory."""
    rng = np.random.default_rng(12)
    batch, next_n, mml, k = 5, 2, 20000, 512
    ctx = np.array([0, 3, 700, 12000, 20000], dtype=np.int32)
    logits = rng.normal(size=(batch * next_n, mml)).astype(np.float32)
    want = gpu_paged_topk(fp8idx, logits, ctx, next_n, mml, k)
    host = torch.full((batch * next_n, k), -7, dtype=torch.int32).pin_memory()
    fp8idx.fp8_paged_topk(torch.from_numpy(logits).cuda(), torch.from_numpy(ctx).cuda(), next_n, mml, k, host)
    torch.cuda.synchronize()
    assert np.array_equal(host.numpy(), want)
    ks, ke = T.decode_windows(ctx, next_n, mml)
    want = gpu_mqa_topk(fp8idx, logits, ks.astype(np.int32), ke.astype(np.int32), k)
    host.fill_(-7)
    fp8idx.fp8_mqa_topk(torch.from_numpy(logits).cuda(), torch.from_numpy(ks.astype(np.int32)).cuda(),
                        torch.from_numpy(ke.astype(np.int32)).cuda(), k, host)
    torch.cuda.synchronize()
    assert np.array_equal(host.numpy(), want)


def test_topk_more_rows_than_sms(fp8idx):
    """More rows than SMs (several waves of CTAs, two per SM): short, long,
    tied and empty windows."""
    rng = np.random.default_rng(21)
    m, n = 400, 24000
    logits = rng.normal(size=(m, n)).astype(np.float32)
    logits[::7] = np.round(logits[::7], 1)
    ks = rng.integers(-100, n, m).astype(np.int32)
    ke = (ks + rng.integers(-50, n, m)).astype(np.int32)
    ks[:20], ke[:20] = 0, n
    for k in (64, 2048):
        want = T.topk_rows(logits, *T.prefill_windows(ks, ke, n), k)
        got = gpu_mqa_topk(fp8idx, logits, ks, ke, k)
        bad = np.nonzero((got != want).any(axis=1))[0]
        assert bad.size == 0, f"k={k} rows {bad[:10].tolist()}"


@pytest.mark.parametrize("ctas", [1, 2, 3, 4, 8])
def test_topk_ctas_per_row(fp8idx, ctas):
    """The same rows split over 1..8 CTAs (2 or more: one thread-block
    cluster per row): windows whose slices fit shared memory, long ones
    (sampled threshold), heavy ties (the exact fallback), a window only a
    few values longer than k, one shorter than k, an empty one."""
    rng = np.random.default_rng(40 + ctas)
    m, n = 10, 150000
    logits = rng.normal(size=(m, n)).astype(np.float32)
    logits[3] = rng.integers(0, 3, n).astype(np.float32)
    logits[4, ::7] = np.round(logits[4, ::7], 1)
    ks = np.array([0, 0, 17, 5, 0, 149990, 0, 3, 100, 0], dtype=np.int32)
    ke = np.array([150000, 9000, 120001, 150000, 150000, 150000, 0, 70003, 2153, 40000], dtype=np.int32)
    for k in (1, 512, 2048):
        want = T.topk_rows(logits, *T.prefill_windows(ks, ke, n), k)
        got = gpu_mqa_topk(fp8idx, logits, ks, ke, k, ctas)
        bad = np.nonzero((got != want).any(axis=1))[0]
        assert bad.size == 0, f"ctas={ctas} k={k} rows {bad.tolist()}"


def test_topk_of_library_logits(fp8idx, oracle_impl):
    """End to end: the decode logits kernel's output feeds the top-k; GPU and
    oracle top-k see the same (GPU) logits."""
    case = workloads.decode_case(4, 2, 32, max_model_len=6000, block_size=64, var_ratio=0.4, seed=3)
    d = to_device(case)
    out = torch.full((8, 6000), float("-inf"), device="cuda")
    fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"], 6000, out)
    idx = torch.empty((8, 2048), dtype=torch.int32, device="cuda")
    fp8idx.fp8_paged_topk(out, d["context_lens"], 2, 6000, 2048, idx)
    torch.cuda.synchronize()
    logits = out.cpu().numpy()
    want = T.topk_rows(logits, *T.decode_windows(case.context_lens, 2, 6000), 2048)
    assert np.array_equal(idx.cpu().numpy(), want)


def test_topk_errors(fp8idx):
    lg = torch.zeros((4, 100), device="cuda")
    idx = torch.empty((4, 10), dtype=torch.int32, device="cuda")
    ks = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(fp8idx.Fp8IdxError) as e:
        fp8idx.fp8_mqa_topk(lg, ks, ks, 4096, torch.empty((4, 4096), dtype=torch.int32, device="cuda"))
    assert e.value.status == fp8idx.FP8IDX_ERR_UNSUPPORTED
    with pytest.raises(fp8idx.Fp8IdxError) as e:
        fp8idx.fp8_mqa_topk(lg, ks, ks, 11, idx)
    assert e.value.status == fp8idx.FP8IDX_ERR_INVALID
    with pytest.raises(fp8idx.Fp8IdxError) as e:
        fp8idx.fp8_paged_topk(lg, ks[:3], 1, 100, 10, idx)
    assert e.value.status == fp8idx.FP8IDX_ERR_INVALID
    with pytest.raises(fp8idx.Fp8IdxError) as e:
        fp8idx.fp8_mqa_topk(lg, ks, ks, 10, idx, ctas_per_row=9)
    assert e.value.status == fp8idx.FP8IDX_ERR_UNSUPPORTED
