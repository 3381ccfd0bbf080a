"""bench.py without a GPU: the reference arm (the CPU oracle) prints one
JSON line with the contract's keys, and the work counts match hand sums."""
import json
import os
import subprocess
import sys

import helpers
import synth

sys.path.insert(0, helpers.ROOT)
import bench  # noqa: E402


def test_reference_arm_prints_contract_line():
    out = subprocess.run([sys.executable, os.path.join(helpers.ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "decode_1x4096", "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, check=True, timeout=300).stdout.strip().splitlines()
    line = json.loads(out[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_work_counts_by_hand():
    w = synth.workload("decode_4x65536")
    wc = bench.work_counts(w)
    # 4 sequences x 65,536 positions x 4 heads x 64 dims x 2 bytes of index keys, plus iq and pooled scores
    assert wc["scan_bytes"] == 4 * (65536 * 4 * 128 + 4 * 128 + 1024 * 4 * 4)
    # kept keys per row and head: 15 full blocks + the local block up to p = 65,535 (64 keys)
    assert wc["dec_att_bytes"] == 4 * (4 * 1024 * 128 * 4 + 64 * 128 * 6)
    w3 = synth.workload("prefill_4096_at_8192")
    wc3 = bench.work_counts(w3)
    kept = sum(15 * 64 + (p % 64) + 1 for p in range(8192, 12288))
    assert wc3["att_flops"] == 4 * 128 * kept * 4 * 16
    assert wc3["idx_flops"] == sum(2 * 64 * (p + 1) * 4 for p in range(8192, 12288))
