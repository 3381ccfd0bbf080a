"""Prompt-chunk path (sequences with several rows: tcgen05 indexer with the
pool and top-k in its epilogue, tcgen05 attention) and mixed batches on the
GPU against the CPU oracle: selections bit-exact, outputs within tolerance."""
import numpy as np
import pytest
import torch

import synth
from gpu_common import (assert_out_close, assert_selection_equal, device_inputs, msa, oracle_forward, problem,
                        run_forward)

pytestmark = pytest.mark.gpu

CHUNKS = [(130, 700), (64, 64), (2, 5), (200, 1300), (129, 4000), (3, 1025), (128, 128)]


@pytest.mark.parametrize("H,G", [(1, 16), (4, 16), (2, 8), (8, 1), (2, 13)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_prefill_forward_chunks(H, G, out_dtype):
    w = synth.Workload("pre_chunks", H=H, G=G, seqs=CHUNKS, seed=100 + H * 7 + G)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x, out_dtype)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], out_dtype)


@pytest.mark.parametrize("top_k", [1, 3, 8, 16])
def test_prefill_forward_top_k(top_k):
    w = synth.Workload("pre_topk", H=4, G=16, seqs=[(300, 2500), (70, 900)], seed=17, top_k=top_k)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_mixed_batch_small():
    """Decode rows and prompt chunks in one call; unknown decode count too."""
    seqs = [(1, 3000), (40, 1200), (1, 65), (1, 1), (257, 3100), (1, 9000)]
    w = synth.Workload("mixed_small", H=4, G=16, seqs=seqs, seed=23)
    x = synth.make_inputs(w)
    ref = oracle_forward(w, x)
    for hint in ("auto", -1):
        out, sel, nsel = run_forward(w, x, num_decode_seqs=hint)
        assert_selection_equal(sel, nsel, ref)
        assert_out_close(out, ref["out"], torch.float32)


def test_prefill_ties_everywhere():
    w = synth.Workload("pre_ties", H=2, G=16, seqs=[(150, 3000)], seed=29)
    x = synth.make_inputs(w)
    x["ik"][:] = x["ik"][0, 0, :]
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_attend_prefill_staged_on_oracle_selection():
    """msa_attend_prefill on the oracle's selection, every row (decode rows
    included: the staged form takes any sequence)."""
    m = msa()
    seqs = [(1, 2000), (90, 1500), (1, 70), (33, 33)]
    w = synth.Workload("pre_staged", H=4, G=16, seqs=seqs, seed=31)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    ref = oracle_forward(w, x)
    out = m.attend_prefill(pb, dx["q"], dx["k"], dx["v"], torch.from_numpy(ref["sel"]).cuda(),
                           torch.from_numpy(ref["nsel"]).cuda())
    torch.cuda.synchronize()
    assert_out_close(out, ref["out"], torch.float32)


def test_prefill_staged_scores_and_selection():
    m = msa()
    w = synth.Workload("pre_stage12", H=2, G=16, seqs=[(100, 1000), (1, 300)], seed=37)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    scores = m.index_scores(pb, dx["iq"], dx["ik"])
    sel, nsel = m.select_blocks(pb, scores)
    ref = oracle_forward(w, x, with_out=False)
    assert_selection_equal(sel, nsel, ref)


def test_prefill_deterministic():
    w = synth.Workload("pre_det", H=4, G=16, seqs=[(500, 6000)], seed=41)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    o1, s1, _ = run_forward(w, x, dx=dx)
    o2, s2, _ = run_forward(w, x, dx=dx)
    assert torch.equal(s1, s2) and torch.equal(o1, o2)


@pytest.mark.parametrize("name", ["prefill_4096_at_8192", "mixed_8dec_512pre"])
def test_prefill_workloads_full_size(name):
    w = synth.workload(name)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_prefill_long_prefix():
    """A 256-row chunk after a 131,072-token prefix: the indexer splits each
    (row tile, head) over position ranges and merges their lists; selections
    reach back over 2,000+ blocks."""
    w = synth.Workload("pre_long", H=4, G=16, seqs=[(256, 131072 + 256)], seed=34)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


@pytest.mark.parametrize("H,seqs,ties", [
    (2, [(2200, 6000)], False),              # 4 position ranges per (row tile, head) on 152 SMs
    (2, [(900, 2000), (33, 2100)], True),    # 4 ranges, every index score equal
    (4, [(700, 3333)], False),               # 5 ranges, ragged row tile and position tail
    (1, [(20, 40000)], False),               # 8 ranges over 157 position tiles
])
def test_prefill_position_splits(H, seqs, ties):
    """The indexer's position ranges: each range keeps its own list of the best
    blocks and the last range to finish merges them all.  With every score
    equal, each range holds its lowest blocks and the merge must still keep
    the lowest overall (ties to the lower block)."""
    w = synth.Workload("pre_splits", H=H, G=16, seqs=seqs, seed=61 + H + len(seqs))
    x = synth.make_inputs(w)
    if ties:
        x["ik"][:] = x["ik"][0, 0, :]
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)
