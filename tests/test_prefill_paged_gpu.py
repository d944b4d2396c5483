"""GPU parity of fp8_mqa_logits_paged (prefill with the K gather from the
paged cache fused into the kernel) against the CPU oracle (the oracle's own
gather, then the prefill oracle), and bit-identity with fp8_mqa_logits on the
gathered K: only the K source differs between the two paths."""
import numpy as np
import pytest
import torch

import oracle
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


def run_paged(fp8idx, case, clean_logits=True, options=None):
    d = to_device(case)
    out = torch.full((case.rows, case.cols), float("nan"), device="cuda")
    fp8idx.fp8_mqa_logits_paged(d["q"], d["kv_cache"], d["block_tables"], d["cu_seq_lens"], d["weights"], d["ks"],
                                d["ke"], out, clean_logits=clean_logits, options=options)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def gathered(case):
    return oracle.gather_paged_k(case.kv_cache, case.block_tables, case.cu_seq_lens, case.block_size,
                                 dim=case.q.shape[2])


@pytest.mark.parametrize("dim", [128, 64])
@pytest.mark.parametrize("blk", [1, 16, 32, 64, 128])
@pytest.mark.parametrize("heads", [32, 64])
def test_paged_prefill_block_sizes(fp8idx, oracle_impl, blk, heads, dim):
    """Every block size (1: the co-packed cache, gathered per token) and both
    head dims of the prefill sweep, against the oracle's own gather, and
    bit-identical to the contiguous kernel on the gathered K."""
    case = workloads.paged_prefill_case([700, 0, 333, 1030, 5], [64, 0, 333, 100, 5], heads, block_size=blk,
                                        dim=dim, seed=blk + heads + dim, poison=True, extra_blocks=7)
    k, s = gathered(case)
    ref = oracle_impl.mqa_logits(case.q, k, s, case.weights, case.ks, case.ke)
    gpu = run_paged(fp8idx, case)
    assert_rows_close(gpu, ref, what=f"blk{blk}/h{heads}")
    # the same K through the contiguous entry point: identical bits
    d = to_device(case)
    out = torch.full((case.rows, case.cols), float("nan"), device="cuda")
    fp8idx.fp8_mqa_logits(d["q"], torch.from_numpy(k).cuda(), torch.from_numpy(s).cuda(), d["weights"], d["ks"],
                          d["ke"], out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), gpu, equal_nan=True)


@pytest.mark.parametrize("split", [0, 1, 4])
def test_paged_prefill_many_small_requests(fp8idx, oracle_impl, split):
    """Tiles that span several requests (lengths well below the 128-token
    tile), with the planner's column split and forced ones."""
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 90, 40)
    rows = np.minimum(lens, rng.integers(0, 6, 40))
    case = workloads.paged_prefill_case(lens, rows, 32, block_size=16, seed=8, poison=True, extra_blocks=2)
    k, s = gathered(case)
    gpu = run_paged(fp8idx, case, options=fp8idx.Options(split_n=split))
    assert_rows_close(gpu, oracle_impl.mqa_logits(case.q, k, s, case.weights, case.ks, case.ke),
                      what=f"small requests split {split}")


@pytest.mark.parametrize("blk", [16, 1])
def test_paged_prefill_max_requests(fp8idx, oracle_impl, blk):
    """The largest request count a call accepts (4096: the request offsets
    and the padded tile prefix live in shared memory), requests of 0 to 7
    tokens with 0 or 1 query rows, against the oracle on every row; one
    request more is UNSUPPORTED."""
    R = 4096
    rng = np.random.default_rng(17)
    lens = rng.integers(0, 8, R)
    rows = np.minimum(lens, rng.integers(0, 2, R))
    case = workloads.paged_prefill_case(lens, rows, 32, block_size=blk, seed=18)
    k, s = gathered(case)
    gpu = run_paged(fp8idx, case)
    assert_rows_close(gpu, oracle_impl.mqa_logits(case.q, k, s, case.weights, case.ks, case.ke),
                      what=f"{R} requests blk{blk}")
    if blk == 16:
        lens2 = np.ones(R + 1, np.int64)
        big = workloads.paged_prefill_case(lens2, lens2, 32, block_size=16, seed=19)
        with pytest.raises(fp8idx.Fp8IdxError) as e:
            run_paged(fp8idx, big)
        assert e.value.status == fp8idx.FP8IDX_ERR_UNSUPPORTED


def test_paged_prefill_no_clean_and_overrides(fp8idx, oracle_impl):
    case = workloads.paged_prefill_case([900, 257], [70, 40], 32, block_size=64, seed=11, poison=True)
    k, s = gathered(case)
    ref = oracle_impl.mqa_logits(case.q, k, s, case.weights, case.ks, case.ke)
    assert_rows_close(run_paged(fp8idx, case, clean_logits=False), ref, written=np.isfinite(ref), what="no-clean")
    for opts in (dict(split_n=1), dict(stages=2), dict(block_m=3, split_n=3), dict(split_n=2), dict(split_n=5),
                 dict(split_n=13)):
        gpu = run_paged(fp8idx, case, options=fp8idx.Options(**opts))
        assert_rows_close(gpu, ref, what=str(opts))
        gpu = run_paged(fp8idx, case, clean_logits=False, options=fp8idx.Options(**opts))
        assert_rows_close(gpu, ref, written=np.isfinite(ref), what=f"no-clean {opts}")


@pytest.mark.slow
def test_paged_prefill_full_size_matches_contiguous(fp8idx):
    """The 4 x 1024-row causal workload over 32768 gathered tokens (block 64):
    bit-identical to the contiguous kernel on the gathered K, which the
    prefill tests check against the oracle at this size -- so every output
    element, the -inf fill of every split included, is covered."""
    case = workloads.paged_prefill_case([8192] * 4, [1024] * 4, 32, block_size=64, seed=77)
    k, s = gathered(case)
    d = to_device(case)
    for split in (0, 1, 3):
        gpu = run_paged(fp8idx, case, options=fp8idx.Options(split_n=split))
        out = torch.full((case.rows, case.cols), float("nan"), device="cuda")
        fp8idx.fp8_mqa_logits(d["q"], torch.from_numpy(k).cuda(), torch.from_numpy(s).cuda(), d["weights"],
                              d["ks"], d["ke"], out)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), gpu, equal_nan=True), f"split {split}"


def test_paged_prefill_errors(fp8idx):
    case = workloads.paged_prefill_case([10], [2], 32, block_size=16, seed=1)
    d = to_device(case)
    out = torch.empty((case.rows, case.cols), device="cuda")
    with pytest.raises(fp8idx.Fp8IdxError) as e:  # cu_seq_lens must have requests + 1 entries
        fp8idx.fp8_mqa_logits_paged(d["q"], d["kv_cache"], d["block_tables"], d["cu_seq_lens"][:1], d["weights"],
                                    d["ks"], d["ke"], out)
    assert e.value.status == fp8idx.FP8IDX_ERR_INVALID
    blk8 = workloads.paged_prefill_case([10], [2], 32, block_size=8, seed=1)
    d8 = to_device(blk8)
    with pytest.raises(fp8idx.Fp8IdxError) as e:  # block size 8: not implemented
        fp8idx.fp8_mqa_logits_paged(d8["q"], d8["kv_cache"], d8["block_tables"], d8["cu_seq_lens"], d8["weights"],
                                    d8["ks"], d8["ke"], torch.empty((blk8.rows, blk8.cols), device="cuda"))
    assert e.value.status == fp8idx.FP8IDX_ERR_UNSUPPORTED
    blk1 = workloads.paged_prefill_case([10], [2], 32, block_size=1, seed=1)
    d1 = to_device(blk1)
    with pytest.raises(fp8idx.Fp8IdxError) as e:  # the token gather needs at least 6 stages
        fp8idx.fp8_mqa_logits_paged(d1["q"], d1["kv_cache"], d1["block_tables"], d1["cu_seq_lens"], d1["weights"],
                                    d1["ks"], d1["ke"], torch.empty((blk1.rows, blk1.cols), device="cuda"),
                                    options=fp8idx.Options(stages=3))
    assert e.value.status == fp8idx.FP8IDX_ERR_UNSUPPORTED


def test_paged_prefill_offsets_past_n_stay_inside_out(fp8idx):
    """cu_seq_lens that break the precondition (a last offset past N, an
    offset that decreases) are clamped on the device into [0, N] and made
    non-decreasing, so no store leaves the output: out is a column slice of a
    wider NaN buffer whose guard columns must stay untouched, and every
    element of [0, N) is written (-inf or a finite logit)."""
    case = workloads.paged_prefill_case([300, 200, 150], [40, 30, 20], 32, block_size=16, seed=12)
    n = case.cols  # 650
    d = to_device(case)
    bad = case.cu_seq_lens.copy()
    bad[2] = bad[1] - 7          # decreasing
    bad[3] = n + 90              # past N
    d["cu_seq_lens"] = torch.from_numpy(bad).cuda()
    pitch = n + 132
    buf = torch.full((case.rows, pitch), float("nan"), device="cuda")
    fp8idx.fp8_mqa_logits_paged(d["q"], d["kv_cache"], d["block_tables"], d["cu_seq_lens"], d["weights"], d["ks"],
                                d["ke"], buf[:, :n])
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    assert np.isnan(host[:, n:]).all(), "a store landed past column N"
    assert not np.isnan(host[:, :n]).any(), "an element of [0, N) was left unwritten"
    assert fp8idx.device_status() == fp8idx.FP8IDX_OK


@pytest.mark.parametrize("dim", [128, 64])
def test_paged_prefill_block1_small_requests_and_overrides(fp8idx, oracle_impl, dim):
    """Block size 1: tiles spanning many short requests, a unit count that
    crosses the Q double buffer many times with one CTA, the minimum stage
    count, and clean_logits off."""
    rng = np.random.default_rng(5 + dim)
    lens = rng.integers(0, 300, 30)
    rows = np.minimum(lens, rng.integers(0, 9, 30))
    case = workloads.paged_prefill_case(lens, rows, 32, block_size=1, dim=dim, seed=9, poison=True, extra_blocks=40)
    k, s = gathered(case)
    ref = oracle_impl.mqa_logits(case.q, k, s, case.weights, case.ks, case.ke)
    for opts in (None, dict(num_ctas=1), dict(stages=6), dict(split_n=3, num_ctas=2)):
        o = fp8idx.Options(**opts) if opts else None
        assert_rows_close(run_paged(fp8idx, case, options=o), ref, what=f"blk1 d{dim} {opts}")
    assert_rows_close(run_paged(fp8idx, case, clean_logits=False), ref, written=np.isfinite(ref),
                      what=f"blk1 d{dim} no-clean")
