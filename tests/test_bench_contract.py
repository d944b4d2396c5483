"""The benchmark's output contract and its recorded ncu traffic (CPU): the
reference arm's JSON line on a small workload, and the structure of the
per-workload DRAM traffic record that `roofline.traffic` is read from."""
import json
import os
import re
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "decode_b1", "--steps", "3",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is False and d["warmup"] >= 3 and d["steps"] == 3
    assert d["config"]["workload"] == "decode_b1"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["value"] > 0


def test_recorded_traffic_structure():
    """One entry per bench workload: a positive byte count, the kernel it was
    taken on, and a 16-hex hash of the sources that build that kernel."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    names = set(bench.WORKLOADS) | set(bench.TOPK_WORKLOADS)
    assert names <= set(rec), names - set(rec)
    kernel_of = {"decode": "paged_logits_kernel", "prefill": "mqa_logits_kernel", "topk": "topk_rows_kernel"}
    for w in names:
        e = rec[w]
        assert isinstance(e["dram_bytes_per_launch"], int) and e["dram_bytes_per_launch"] > 0, w
        assert re.fullmatch(r"[0-9a-f]{16}", e["kernel_hash"]), w
        assert e["kernel"].startswith(kernel_of[bench.workload_kernel(w)]), w


def test_kernel_hash_covers_the_kernel_and_shared_sources():
    """Workloads of one kernel share a hash; different kernels differ; a
    figure is reported only when the recorded hash matches."""
    h = {w: bench.kernel_source_hash(w) for w in ("decode_mtp_verify", "decode_b1", "prefill_4x1024",
                                                  "prefill_paged_4x1024", "topk_decode_mtp_verify")}
    assert h["decode_mtp_verify"] == h["decode_b1"]
    assert h["prefill_4x1024"] == h["prefill_paged_4x1024"]
    assert len({h["decode_mtp_verify"], h["prefill_4x1024"], h["topk_decode_mtp_verify"]}) == 3
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for w in h:
        got = bench.recorded_traffic(w)
        assert got == (rec[w]["dram_bytes_per_launch"] if rec[w]["kernel_hash"] == h[w] else None)
