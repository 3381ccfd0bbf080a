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


def test_rotation_sets_clear_the_l2():
    """Back-to-back timing rotates enough input copies that the other copies'
    bytes between two uses of one copy exceed twice the L2; tiny workloads
    fall back to the flush."""
    for name in synth.WORKLOADS:
        w = synth.workload(name)
        n = bench.rotation_sets(w)
        t = bench.step_touched_bytes(w)
        if n:
            assert 3 <= n <= 8
            assert (n - 1) * t > 2 * bench.L2_BYTES, (name, n, t)
        else:
            assert 7 * t <= 2 * bench.L2_BYTES, (name, t)
    assert bench.rotation_sets(synth.workload("decode_1x4096")) == 0
    assert bench.rotation_sets(synth.workload("decode_4x65536")) == 3


def test_step_touched_bytes_by_hand():
    w = synth.workload("prefill_4096_at_8192")
    # q in (bf16) and out (fp32) of 4,096 rows x 64 heads x 128 dims, iq, and the causal caches (ik 64 + k, v 128 dims)
    want = 4096 * 64 * 128 * 6 + 4096 * 4 * 64 * 2 + 12288 * (4 * 64 + 2 * 4 * 128) * 2
    assert bench.step_touched_bytes(w) == want
    w2 = synth.workload("decode_4x65536")
    wc = bench.work_counts(w2)
    assert bench.step_touched_bytes(w2) == wc["scan_bytes"] + wc["dec_att_bytes"]


def test_timing_fields_pick_back_to_back_when_measured():
    res = {"ms_per_step": 0.040, "b2b_ms_per_step": 0.034, "b2b_sets": 3}
    assert bench.step_ms(res) == 0.034
    assert "rotating" in bench.timing_note(res)
    lat = bench.flushed_latency(res, rows=4, ws=1)
    assert lat["ms_per_step"] == 0.04 and abs(lat["value"] - 100000.0) < 1e-6
    flushed_only = {"ms_per_step": 0.017}
    assert bench.step_ms(flushed_only) == 0.017
    assert bench.flushed_latency(flushed_only, rows=1, ws=1) is None
    assert "flushed" in bench.timing_note(flushed_only)
