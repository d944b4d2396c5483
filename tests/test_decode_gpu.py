"""GPU parity of fp8_paged_mqa_logits (decode) against the CPU oracle.

Every case NaN-poisons the output, so a window position the kernel fails to
write, or a position outside the window it writes, is caught (decode writes
only the causal window; the -inf outside is the caller's).  Block tables
point into a permuted pool with NaN-poisoned unowned blocks and tail slots,
so a kernel that walks the cache linearly or reads past a context fails.
"""
import zlib

import numpy as np
import pytest
import torch

import workloads
from parity import assert_rows_close, decode_window_mask, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8idx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_fp8_gb300 as m
    m.library()
    return m


def run_decode(fp8idx, case, options=None, out=None):
    d = to_device(case)
    rows = case.batch * case.next_n
    if out is None:
        out = torch.full((rows, case.max_model_len), float("nan"), dtype=torch.float32, device="cuda")
    fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                case.max_model_len, out, options=options)
    torch.cuda.synchronize()
    return out


def oracle_decode(o, case, rows=None):
    return o.paged_mqa_logits(case.q, case.kv_cache, case.weights, case.context_lens, case.block_tables,
                              case.block_size, case.max_model_len, rows=rows)


SMALL = [
    # (name, batch, next_n, heads, max_model_len, block_size, context_lens)
    ("b1_n1_h32_blk64_full", 1, 1, 32, 1024, 64, [1024]),
    ("b3_n2_h32_blk64_ragged", 3, 2, 32, 700, 64, [700, 129, 1]),
    ("b4_n6_h32_blk64_short", 4, 6, 32, 600, 64, [600, 255, 5, 6]),
    ("b2_n8_h32_blk16", 2, 8, 32, 300, 16, [300, 77]),
    ("b2_n4_h64_blk32", 2, 4, 64, 520, 32, [520, 300]),
    ("b5_n3_h64_blk128", 5, 3, 64, 400, 128, None),
    ("b3_n5_h32_blk64", 3, 5, 32, 450, 64, [450, 128, 127]),
    ("b3_n4_h64_blk1", 3, 4, 64, 333, 1, [333, 200, 4]),
    ("b2_n2_h32_blk1_ctx0", 2, 2, 32, 900, 1, [900, 0]),
    ("b2_n1_h64_blk64_ctx0", 2, 1, 64, 256, 64, [0, 256]),
    ("b6_n1_h32_blk1_ragged", 6, 1, 32, 1000, 1, None),
]


@pytest.mark.parametrize("name,batch,next_n,heads,mml,blk,ctx", SMALL, ids=[s[0] for s in SMALL])
def test_decode_small(fp8idx, oracle_impl, name, batch, next_n, heads, mml, blk, ctx):
    case = workloads.decode_case(batch, next_n, heads, max_model_len=mml, block_size=blk, context_lens=ctx,
                                 var_ratio=0.3, seed=zlib.crc32(name.encode()) % 1000, poison=True, extra_blocks=3)
    gpu = run_decode(fp8idx, case).cpu().numpy()
    ref = oracle_decode(oracle_impl, case)
    assert_rows_close(gpu, ref, written=decode_window_mask(case), what=name)


@pytest.mark.parametrize("opts", [dict(num_ctas=1), dict(num_ctas=3), dict(stages=2), dict(stages=3, num_ctas=5),
                                  dict(stages=6, num_ctas=2)],
                         ids=["one_cta", "three_ctas", "two_stages", "three_stages", "gather_min_stages"])
def test_decode_planner_overrides(fp8idx, oracle_impl, opts):
    """One CTA crossing many requests exercises the Q/weight double buffer and
    every ring wrap; small stage counts exercise the back-pressure paths."""
    blk = 1 if opts.get("stages") == 6 else 64
    case = workloads.decode_case(7, 3, 32, max_model_len=520, block_size=blk, var_ratio=0.6, seed=7,
                                 poison=True, extra_blocks=2)
    gpu = run_decode(fp8idx, case, options=fp8idx.Options(**opts)).cpu().numpy()
    ref = oracle_decode(oracle_impl, case)
    assert_rows_close(gpu, ref, written=decode_window_mask(case), what=str(opts))


@pytest.mark.parametrize("num_ctas", [1, 2, 5, 0])
def test_decode_block1_table_prefetch_edges(fp8idx, oracle_impl, num_ctas):
    """Block size 1: each producer lane loads its block-table entries two
    tiles ahead of their use.  Requests of 1 token to 5 tiles, one exactly a
    tile long, and CTA ranges that start inside a request (num_ctas) cover
    every case of that look-ahead: a request shorter than the look-ahead,
    the last tiles of a request, and a range that begins mid-request."""
    ctx = [1, 129, 256, 257, 383, 130, 2, 640]
    case = workloads.decode_case(len(ctx), 2, 32, max_model_len=640, block_size=1, context_lens=ctx, seed=71,
                                 poison=True, extra_blocks=3)
    opts = fp8idx.Options(num_ctas=num_ctas) if num_ctas else None
    gpu = run_decode(fp8idx, case, options=opts).cpu().numpy()
    ref = oracle_decode(oracle_impl, case)
    assert_rows_close(gpu, ref, written=decode_window_mask(case), what=f"blk1 num_ctas={num_ctas}")


@pytest.mark.parametrize("blk", [64, 1])
def test_decode_max_batch(fp8idx, oracle_impl, blk):
    """The largest batch a call accepts (4096 requests: the per-request tile
    prefix lives in shared memory and the planner trims the ring for it),
    with short ragged contexts (0 to 300 tokens), against the oracle on every
    row; one request more is UNSUPPORTED."""
    B = 4096
    rng = np.random.default_rng(91)
    ctx = rng.integers(0, 301, size=B)
    ctx[:3] = [0, 1, 300]
    case = workloads.decode_case(B, 2, 32, max_model_len=320, block_size=blk, context_lens=ctx, seed=91)
    gpu = run_decode(fp8idx, case).cpu().numpy()
    ref = oracle_decode(oracle_impl, case)
    assert_rows_close(gpu, ref, written=decode_window_mask(case), what=f"batch {B} blk{blk}")
    if blk == 64:
        big = workloads.decode_case(B + 1, 1, 32, max_model_len=64, block_size=64, context_lens=[64] * (B + 1), seed=92)
        with pytest.raises(fp8idx.Fp8IdxError) as e:
            run_decode(fp8idx, big)
        assert e.value.status == fp8idx.FP8IDX_ERR_UNSUPPORTED


def test_decode_into_pinned_host_memory(fp8idx):
    """A pinned host tensor as the output: the kernel writes the windows
    straight into host memory (through its device mapping), bit for bit what
    it writes into device memory, and leaves the rest untouched."""
    case = workloads.decode_case(3, 2, 32, max_model_len=700, block_size=64, context_lens=[700, 300, 5], seed=5,
                                 poison=True, extra_blocks=1)
    dev = run_decode(fp8idx, case).cpu().numpy()
    host = torch.full(dev.shape, float("nan"), dtype=torch.float32).pin_memory()
    d = to_device(case)
    fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                case.max_model_len, host)
    torch.cuda.synchronize()
    assert np.array_equal(host.numpy(), dev, equal_nan=True)
    with pytest.raises(ValueError, match="pinned"):
        fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                    case.max_model_len, torch.empty(dev.shape, dtype=torch.float32))
    with pytest.raises(ValueError, match="inputs must be CUDA"):
        fp8idx.fp8_paged_mqa_logits(d["q"].cpu(), d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                    case.max_model_len, host)


def test_decode_config0(fp8idx, oracle_impl):
    case = workloads.make_config(0)
    gpu = run_decode(fp8idx, case).cpu().numpy()
    assert_rows_close(gpu, oracle_decode(oracle_impl, case), written=decode_window_mask(case), what="config0")


def test_decode_config1(fp8idx, oracle_impl):
    case = workloads.make_config(1)
    gpu = run_decode(fp8idx, case).cpu().numpy()
    assert_rows_close(gpu, oracle_decode(oracle_impl, case), written=decode_window_mask(case), what="config1")


def _full_size_dense(fp8idx, o, case, chunk_rows=16):
    """Full-size run in the bench's launch configuration, compared with the
    oracle element by element: every row, streamed through the oracle in
    chunks of rows, each finite logit against its own row's oracle maximum,
    and the written/untouched mask of every element."""
    out = run_decode(fp8idx, case)
    gpu = out.cpu().numpy()
    del out
    nrows = case.batch * case.next_n
    for r0 in range(0, nrows, chunk_rows):
        r1 = min(nrows, r0 + chunk_rows)
        ref = oracle_decode(o, case, rows=(r0, r1))
        assert_rows_close(gpu[r0:r1], ref, written=decode_window_mask(case, rows=(r0, r1)), what=f"rows {r0}..{r1}")


@pytest.mark.slow
def test_decode_config2_full_size(fp8idx, oracle_impl):
    _full_size_dense(fp8idx, oracle_impl, workloads.make_config(2))


@pytest.mark.slow
def test_decode_config2_next_n1_full_size(fp8idx, oracle_impl):
    _full_size_dense(fp8idx, oracle_impl, workloads.make_config(2, next_n=1))


@pytest.mark.slow
def test_decode_config4_full_size(fp8idx, oracle_impl):
    _full_size_dense(fp8idx, oracle_impl, workloads.make_config(4), chunk_rows=32)


def test_decode_graph_capture_replay(fp8idx, oracle_impl):
    """Captured once, replayed with new input contents: matches the oracle."""
    case = workloads.decode_case(4, 2, 32, max_model_len=640, block_size=64, var_ratio=0.3, seed=31,
                                 poison=True, extra_blocks=1)
    d = to_device(case)
    out = torch.full((8, 640), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up on the capture stream
        fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                    640, out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"],
                                    640, out, stream=s)
    case2 = workloads.decode_case(4, 2, 32, max_model_len=640, block_size=64, var_ratio=0.3, seed=32,
                                  poison=True, extra_blocks=1)
    # same shapes; new contents copied into the captured buffers
    case2.context_lens[:] = case.context_lens
    case2.block_tables[:] = case.block_tables
    case2.kv_cache = case.kv_cache
    d["q"].copy_(torch.from_numpy(case2.q))
    d["weights"].copy_(torch.from_numpy(case2.weights))
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    ref = oracle_decode(oracle_impl, case2)
    assert_rows_close(out.cpu().numpy(), ref, written=decode_window_mask(case2), what="graph replay")


def test_decode_empty_and_errors(fp8idx):
    case = workloads.decode_case(2, 2, 32, max_model_len=128, block_size=64, context_lens=[128, 64], seed=3)
    d = to_device(case)
    out = torch.full((4, 128), float("nan"), device="cuda")
    # max_model_len 0: nothing to do
    fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"], 0, out)
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    with pytest.raises(fp8idx.Fp8IdxError) as e:  # weights with the wrong dtype
        fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"].to(torch.int32), d["context_lens"],
                                    d["block_tables"], 128, out)
    assert e.value.status == fp8idx.FP8IDX_ERR_INVALID
    q16 = torch.zeros((2, 2, 16, 128), dtype=torch.uint8, device="cuda")
    w16 = torch.zeros((4, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(fp8idx.Fp8IdxError) as e:  # 16 heads: not implemented
        fp8idx.fp8_paged_mqa_logits(q16, d["kv_cache"], w16, d["context_lens"], d["block_tables"], 128, out)
    assert e.value.status == fp8idx.FP8IDX_ERR_UNSUPPORTED
    assert fp8idx.device_status() == fp8idx.FP8IDX_OK


def test_decode_context_past_table_capacity(fp8idx, oracle_impl):
    """A context longer than the block table can address (a broken
    precondition) is clamped to the table's capacity on the device: the
    kernel stores exactly the window of the clamped context -- what its
    producers loaded -- and nothing past it."""
    cap = 256
    case = workloads.decode_case(3, 2, 32, max_model_len=cap, block_size=64, context_lens=[cap, 200, 130], seed=44,
                                 poison=True, extra_blocks=2)
    ref = oracle_decode(oracle_impl, case)  # the clamped contexts: [256, 200, 130]
    d = to_device(case)
    mml = 512
    d["context_lens"] = torch.tensor([400, 200, 130], dtype=torch.int32, device="cuda")
    out = torch.full((6, mml), float("nan"), device="cuda")
    fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"], mml, out)
    torch.cuda.synchronize()
    gpu = out.cpu().numpy()
    assert np.isnan(gpu[:, cap:]).all(), "positions past the table capacity were stored"
    assert_rows_close(gpu[:, :cap], ref, written=decode_window_mask(case), what="clamped context")
    assert fp8idx.device_status() == fp8idx.FP8IDX_OK
