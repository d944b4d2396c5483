"""The benchmark's byte model against figures the indexer pages print (CPU)."""
import json
import os

import bench

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def test_shared_walk_and_per_row_programs():
    ctx = [131072] * 16
    shared = bench.decode_bytes(16, 6, 32, ctx, 1048576)["total"] / 1e6
    per_row = bench.decode_bytes(16, 6, 32, ctx, 1048576, k_reads=6)["total"] / 1e6
    assert abs(shared - GOLD["shared_k_walk_mb"]["value"]) < 1.0, shared
    assert abs(per_row - GOLD["per_next_n_programs_mb"]["value"]) < 1.0, per_row


def test_decode_output_shape_matches_the_fill():
    g = GOLD["decode_prefill_fill_mb"]
    rows = g["batch"] * g["next_n"]
    fill_mb = rows * g["max_model_len"] * 4 / 1e6  # [batch*next_n, max_model_len] f32
    assert abs(fill_mb - g["value"]) < 0.05
    assert abs(2 * fill_mb - GOLD["nan_to_num_mb"]["value"]) < 0.1


def test_prefill_chunks_share_one_logits_budget():
    outs = {bench.prefill_bytes(m, n, 32)["out"] for m, n in GOLD["prefill_chunk_shapes"]["value"]}
    assert outs == {512 << 20}


def test_window_and_flops():
    # next_n 2, ctx 5: rows see positions 0..3 and 0..4 -> 9 logits
    assert bench.decode_window_elems([5], 2, 100) == 9
    assert bench.decode_window_elems([1], 3, 100) == 1
    assert bench.decode_window_elems([0], 1, 100) == 0
    assert bench.decode_flops(32, [5], 2, 100) == 9 * 2 * 128 * 32
    assert bench.prefill_window_pairs([0, -5, 10], [3, 2, 5], 100) == 3 + 2 + 0
