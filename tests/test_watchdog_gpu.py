"""The bounded-wait watchdog on the GPU: a wait that nothing satisfies runs
out, the kernel returns, the device status reports the timeout with the
waiting site, the status clears, and the device stays usable (a decode call
afterwards still matches the oracle).  The failure is made by a barrier that
nothing arrives on, given a limit of a few milliseconds; no fault, trap or
endless loop is involved."""
import time

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


def test_wait_runs_out_and_device_recovers(fp8idx, oracle_impl):
    torch.cuda.synchronize()
    assert fp8idx.device_status() == fp8idx.FP8IDX_OK  # (also clears)
    try:
        t0 = time.perf_counter()
        fp8idx.watchdog_selftest(5000)  # give up after 5 ms
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert elapsed < 1.0, f"the self-test kernel took {elapsed:.3f} s"
        assert fp8idx.device_status(clear=False) == fp8idx.FP8IDX_ERR_TIMEOUT
        msg = fp8idx.device_status_message()
        assert "decode sites 0x80" in msg, msg
        assert fp8idx.device_status(clear=True) == fp8idx.FP8IDX_ERR_TIMEOUT  # read, then clear
    finally:
        fp8idx.device_status(clear=True)
    assert fp8idx.device_status() == fp8idx.FP8IDX_OK

    case = workloads.decode_case(3, 2, 32, max_model_len=700, block_size=64, var_ratio=0.3, seed=17, poison=True,
                                 extra_blocks=2)
    d = to_device(case)
    out = torch.full((6, 700), float("nan"), device="cuda")
    fp8idx.fp8_paged_mqa_logits(d["q"], d["kv_cache"], d["weights"], d["context_lens"], d["block_tables"], 700, out)
    torch.cuda.synchronize()
    ref = oracle_impl.paged_mqa_logits(case.q, case.kv_cache, case.weights, case.context_lens, case.block_tables,
                                       64, 700)
    assert_rows_close(out.cpu().numpy(), ref, written=decode_window_mask(case), what="decode after the timeout")
    assert fp8idx.device_status() == fp8idx.FP8IDX_OK
