"""Pins of the oracle's paged-K gather (oracle.gather_paged_k), the input of
the fused paged prefill.  Checked against bytes placed by hand, and against
the C oracle's decode path, which walks the block table on its own: a
prefill row over a request's gathered columns equals the decode row of that
request with the same Q and weights (next_n = 1)."""
import numpy as np

import oracle
import workloads


def test_gather_hand_case():
    dim, blk = 4, 2
    page = blk * (dim + 4)
    cache = np.zeros((3, page), np.uint8)
    for b in range(3):
        for slot in range(blk):
            cache[b, slot * dim:(slot + 1) * dim] = 10 * b + slot  # every byte of the row tells (block, slot)
            cache[b, blk * dim + 4 * slot: blk * dim + 4 * slot + 4] = np.array([b + slot / 10], np.float32).view(np.uint8)
    tables = np.array([[2, 0], [1, -1]], np.int32)
    cu = np.array([0, 3, 4], np.int32)
    k, s = oracle.gather_paged_k(cache, tables, cu, blk, dim)
    # request 0: tokens 0,1 from block 2 slots 0,1, token 2 from block 0 slot 0; request 1: block 1 slot 0
    assert k[:, 0].tolist() == [20, 21, 0, 10]
    assert (k == k[:, :1]).all()
    assert np.allclose(s, [2.0, 2.1, 0.0, 1.0])


def test_gather_matches_decode_walk(oracle_impl):
    case = workloads.paged_prefill_case([300, 0, 129, 64], [1, 0, 1, 1], 32, block_size=16, seed=4, poison=True,
                                        extra_blocks=5)
    k, s = oracle.gather_paged_k(case.kv_cache, case.block_tables, case.cu_seq_lens, 16)
    assert not np.isnan(s).any()  # poisoned slots are never gathered
    lens = np.diff(case.cu_seq_lens)
    pre = oracle_impl.mqa_logits(case.q, k, s, case.weights, case.ks, case.ke)
    # decode rows with the same Q / weights: one decode request per prefill row
    reqs = [r for r in range(lens.size) if lens[r] > 0]
    q_dec = case.q[:, None]                      # [M, 1, H, D]
    ctx = np.array([lens[r] for r in reqs], np.int32)
    dec = oracle_impl.paged_mqa_logits(q_dec, case.kv_cache, case.weights, ctx, case.block_tables[reqs], 16,
                                       int(lens.max()))
    for m, r in enumerate(reqs):
        a, b = case.cu_seq_lens[r], case.cu_seq_lens[r + 1]
        assert np.array_equal(pre[m, a:b], dec[m, :b - a]), f"request {r}"
