"""GPU parity of the fused decode logits + top-k (fp8_paged_mqa_topk).

The fused call must return exactly what the unfused pipeline returns: the
top-k (oracle/topk.py: value descending, lowest positions first among equal
values, listed by position, -1 past the window) of the logits that
fp8_paged_mqa_logits writes -- the filter pass forms every logit with the
same arithmetic, so the two see identical values.  The cases cover windows
shorter than k, empty windows, every k the pages use, both item sizes, the
block-size-1 gather, heavy ties at the threshold, and rows whose sample
misleads the threshold in both directions (too high: too few candidates;
too low: more candidates than the cap), which the exact fallback must
resolve."""
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


def item_tokens(case):
    """Tokens per item of the decode kernel (two 128-token tiles when
    next_n*heads <= 128 and the cache is paged by blocks, else one)."""
    return 256 if case.next_n * case.heads <= 128 and case.block_size > 1 else 128


def scale_tokens(case, positions_of_request):
    """Multiplies the K scale of chosen tokens (positive homogeneity: their
    logits scale by the same factor).  positions_of_request(b, ctx) -> (idx, factor)."""
    kv = case.kv_cache.copy()
    blk = case.block_size
    for b in range(case.batch):
        ctx = int(case.context_lens[b])
        pos, factor = positions_of_request(b, ctx)
        for p in pos:
            blk_id = int(case.block_tables[b, p // blk])
            off = blk * 128 + 4 * (p % blk)
            s = kv[blk_id, off:off + 4].view(np.float32)[0] * np.float32(factor)
            kv[blk_id, off:off + 4] = np.frombuffer(np.float32(s).tobytes(), np.uint8)
    case.kv_cache = kv
    return case


def run_both(fp8idx, case, k, options=None):
    d = to_device(case)
    rows = case.batch * case.next_n
    logits = torch.full((rows, case.max_model_len), float("-inf"), device="cuda")
    fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                case.max_model_len, logits, options=options)
    got = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    fp8idx.fp8_paged_mqa_topk(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                              case.max_model_len, k, got, options=options)
    unfused = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    fp8idx.fp8_paged_topk(logits, d["context_lens"], case.next_n, case.max_model_len, k, unfused)
    torch.cuda.synchronize()
    want = T.topk_rows(logits.cpu().numpy(), *T.decode_windows(case.context_lens, case.next_n, case.max_model_len),
                       k)
    return got.cpu().numpy(), want, unfused.cpu().numpy()


CASES = [
    # (name, batch, next_n, heads, mml, blk, context_lens)
    ("b3_n2_h32_blk64", 3, 2, 32, 20000, 64, [20000, 9000, 3000]),
    ("b2_n6_h32_blk16", 2, 6, 32, 40000, 16, [40000, 17000]),
    ("b2_n4_h64_blk1", 2, 4, 64, 12000, 1, [12000, 5000]),
    ("b4_n1_h32_blk128_short", 4, 1, 32, 5000, 128, [5000, 1500, 700, 0]),
    ("b3_n3_h64_blk32", 3, 3, 64, 9000, 32, [9000, 2, 4100]),
]


@pytest.mark.parametrize("k", [1, 7, 512, 2048])
@pytest.mark.parametrize("name,batch,next_n,heads,mml,blk,ctx", CASES, ids=[c[0] for c in CASES])
def test_fused_topk_matches_unfused(fp8idx, name, batch, next_n, heads, mml, blk, ctx, k):
    case = workloads.decode_case(batch, next_n, heads, max_model_len=mml, block_size=blk, context_lens=ctx,
                                 seed=len(name) * 31 + k, poison=True, extra_blocks=3)
    got, want, unfused = run_both(fp8idx, case, k)
    assert np.array_equal(unfused, want), "unfused top-k differs from the oracle on the same logits"
    assert np.array_equal(got, want), f"{name} k={k}: {int((got != want).sum())} indices differ"
    assert fp8idx.device_status() == fp8idx.FP8IDX_OK


def test_fused_topk_all_equal_logits(fp8idx):
    """Every logit 0 (all K scales 0): the threshold equals every value, all
    positions tie and the lowest k positions win (every position is a
    candidate, more than the candidate capacity: the exact fallback)."""
    case = workloads.decode_case(3, 2, 32, max_model_len=9000, block_size=64, context_lens=[9000, 3000, 100], seed=4)
    case = scale_tokens(case, lambda b, ctx: (range(ctx), 0.0))
    for k in (1, 100, 2048):
        got, want, _ = run_both(fp8idx, case, k)
        assert np.array_equal(got, want), f"k={k}"


def test_fused_topk_repeated_keys(fp8idx):
    """Few distinct logits per row: the K rows of each request repeat a
    handful of tokens, so long runs of equal values sit at and above the
    threshold."""
    case = workloads.decode_case(2, 2, 32, max_model_len=16000, block_size=16, context_lens=[16000, 7000], seed=9)
    kv = case.kv_cache.copy()
    blk = case.block_size
    for b in range(case.batch):
        src = [int(case.block_tables[b, j]) for j in range(3)]
        for j in range(3, -(-int(case.context_lens[b]) // blk)):
            kv[int(case.block_tables[b, j])] = kv[src[j % 3]]
    case.kv_cache = kv
    for k in (7, 512, 2048):
        got, want, _ = run_both(fp8idx, case, k)
        assert np.array_equal(got, want), f"k={k}"


def test_fused_topk_misleading_samples(fp8idx):
    """Sampled items (every 32nd) with scales x50: the threshold from the
    sample sits above almost every other logit, too few candidates pass, and
    the row must take the exact fallback.  Then the opposite: the unsampled
    items x50, the threshold far too low, more candidates than the cap."""
    for boost_sampled in (True, False):
        case = workloads.decode_case(2, 2, 32, max_model_len=60000, block_size=64, context_lens=[60000, 41000],
                                     seed=21)
        it = item_tokens(case)

        def pick(b, ctx, it=it, boost_sampled=boost_sampled):
            pos = [p for p in range(ctx) if ((p // it) % 32 == 0) == boost_sampled]
            return pos, 50.0
        case = scale_tokens(case, pick)
        for k in (512, 2048):
            got, want, _ = run_both(fp8idx, case, k)
            assert np.array_equal(got, want), f"boost_sampled={boost_sampled} k={k}"
    assert fp8idx.device_status() == fp8idx.FP8IDX_OK


def test_fused_topk_planner_overrides_and_graph(fp8idx):
    """A few CTAs crossing requests, and the six launches captured in a CUDA
    graph and replayed with new query contents."""
    case = workloads.decode_case(5, 2, 32, max_model_len=7000, block_size=64, var_ratio=0.5, seed=8, poison=True,
                                 extra_blocks=2)
    got, want, _ = run_both(fp8idx, case, 512, options=fp8idx.Options(num_ctas=3, stages=3))
    assert np.array_equal(got, want)
    d = to_device(case)
    rows, k = case.batch * case.next_n, 512
    ws = torch.empty(fp8idx.paged_mqa_topk_workspace(case.batch, case.next_n, case.max_model_len, k) + 256,
                     dtype=torch.uint8, device="cuda")
    idx = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fp8idx.fp8_paged_mqa_topk(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                  case.max_model_len, k, idx, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fp8idx.fp8_paged_mqa_topk(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                  case.max_model_len, k, idx, workspace=ws, stream=s)
    case2 = workloads.decode_case(5, 2, 32, max_model_len=7000, block_size=64, var_ratio=0.5, seed=8, poison=True,
                                  extra_blocks=2)
    case2.q = workloads.decode_case(5, 2, 32, max_model_len=7000, block_size=64, seed=99).q
    d["q"].copy_(torch.from_numpy(case2.q))
    idx.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    _, want2, _ = run_both(fp8idx, case2, k)
    assert np.array_equal(idx.cpu().numpy(), want2)


def test_fused_topk_errors(fp8idx):
    case = workloads.decode_case(2, 2, 32, max_model_len=512, block_size=64, context_lens=[512, 100], seed=3)
    d = to_device(case)
    idx = torch.empty((4, 64), dtype=torch.int32, device="cuda")
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8idx.Fp8IdxError) as e:  # workspace too small
        fp8idx.fp8_paged_mqa_topk(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"], 512, 64,
                                  idx, workspace=small)
    assert e.value.status == fp8idx.FP8IDX_ERR_INVALID
    with pytest.raises(fp8idx.Fp8IdxError) as e:  # k above 2048
        fp8idx.fp8_paged_mqa_topk(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"], 512,
                                  4096, torch.empty((4, 4096), dtype=torch.int32, device="cuda"))
    assert e.value.status == fp8idx.FP8IDX_ERR_UNSUPPORTED


@pytest.mark.slow
def test_fused_topk_mtp_verify_full_size(fp8idx):
    """The MTP-verify decode batch (16 x next_n 6, 131072-token contexts) at
    k = 2048 and 512: identical to the unfused pipeline."""
    case = workloads.make_config(2)
    for k in (2048, 512):
        got, want, _ = run_both(fp8idx, case, k)
        assert np.array_equal(got, want), f"k={k}: {int((got != want).sum())} indices differ"
