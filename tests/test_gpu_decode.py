"""Decode path (one row per sequence) on the GPU against the CPU oracle:
selections bit-exact, outputs within tolerance; fused and staged entry
points; the decode workloads at full size."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import (assert_out_close, assert_selection_equal, device_inputs, msa, oracle_forward, problem,
                        run_forward)

pytestmark = pytest.mark.gpu

RAGGED = [1, 5, 63, 64, 65, 127, 128, 1000, 1023, 1024, 1025, 4097, 5000, 960, 961]


@pytest.mark.parametrize("H,G", [(1, 16), (2, 16), (4, 16), (8, 4), (4, 1), (2, 7)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_forward_ragged(H, G, out_dtype):
    w = synth.Workload("dec_ragged", H=H, G=G, seqs=[(1, L) for L in RAGGED], seed=H * 31 + G)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x, out_dtype)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], out_dtype)


@pytest.mark.parametrize("top_k", [1, 2, 5, 16])
def test_decode_forward_top_k(top_k):
    w = synth.Workload("dec_topk", H=4, G=16, seqs=[(1, L) for L in [70, 700, 3000, 9000]], seed=7, top_k=top_k)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_decode_ties_everywhere():
    """All index keys equal: every pooled score ties, the lowest blocks win."""
    w = synth.Workload("dec_ties", H=2, G=16, seqs=[(1, 5000), (1, 130)], seed=3)
    x = synth.make_inputs(w)
    x["ik"][:] = x["ik"][0, 0, :]
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    J = (5000 - 1) // 64
    assert sel[0, 0, :].tolist() == list(range(15)) + [J]
    assert_out_close(out, ref["out"], torch.float32)


def test_decode_staged_stages():
    """msa_index_scores exact, msa_select_blocks bit-exact, msa_attend_decode
    on the oracle's selection within tolerance."""
    m = msa()
    w = synth.Workload("dec_staged", H=4, G=16, seqs=[(1, L) for L in [1, 64, 65, 2000, 7777]], seed=11)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    scores = m.index_scores(pb, dx["iq"], dx["ik"])
    pr = oracle.Problem.from_workload(w, x)
    sc = scores.cpu().numpy()
    for r in range(pb.total_rows):
        for h in range(w.H):
            ref = oracle.index_scores(pr, x["iq"], x["ik"], r, h)
            assert np.array_equal(sc[r, h, :len(ref)], ref.astype(np.float32))
            assert np.all(np.isneginf(sc[r, h, len(ref):]))
    sel, nsel = m.select_blocks(pb, scores)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    sel_o = torch.from_numpy(ref["sel"]).cuda()
    nsel_o = torch.from_numpy(ref["nsel"]).cuda()
    out = m.attend_decode(pb, dx["q"], dx["k"], dx["v"], sel_o, nsel_o)
    torch.cuda.synchronize()
    assert_out_close(out, ref["out"], torch.float32)


BATCH40 = [70, 300, 1000, 1100, 2000, 3000, 5000, 9000, 64, 129]


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_decode_clusters_of_four(kv):
    """40 (row, KV head) problems, more than the clusters of 8 CTAs that fit
    on the GPU at once: the attention takes clusters of 4 CTAs, each CTA two
    rounds of two kept blocks with the softmax carried over between them
    (short rows leave CTAs with one block or none).  Fused path, and the
    given selection with bf16 output, against the oracle."""
    m = msa()
    w = synth.Workload("dec_cl4", H=4, G=16, seqs=[(1, L) for L in BATCH40], seed=41, kv_dtype=kv)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)
    dx = device_inputs(x)
    pb = problem(w, x, torch.bfloat16)
    out_g = m.attend_decode(pb, dx["q"], dx["k"], dx["v"], torch.from_numpy(ref["sel"]).cuda(),
                            torch.from_numpy(ref["nsel"]).cuda())
    torch.cuda.synchronize()
    assert_out_close(out_g, ref["out"], torch.bfloat16)


def test_decode_attend_given_selection_any_blocks():
    """A synthetic (not top-k) selection: attention follows the given list."""
    m = msa()
    w = synth.Workload("dec_given", H=2, G=16, seqs=[(1, 3000), (1, 700)], seed=5, top_k=4)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    sel = np.array([[[0, 7, 20, 46], [3, 4, 5, 46]], [[1, 10, -1, -1], [10, -1, -1, -1]]], dtype=np.int32)
    nsel = np.array([[4, 4], [2, 1]], dtype=np.int32)
    out = m.attend_decode(pb, dx["q"], dx["k"], dx["v"], torch.from_numpy(sel).cuda(), torch.from_numpy(nsel).cuda())
    torch.cuda.synchronize()
    pr = oracle.Problem.from_workload(w, x)
    o = out.cpu().numpy()
    for r in range(2):
        for h in range(2):
            ref = oracle.attend(pr, x["q"], x["k"], x["v"], r, h, sel[r, h, :nsel[r, h]])
            assert np.abs(o[r, h * 16:(h + 1) * 16] - ref).max() <= 2e-3


def test_decode_deterministic():
    w = synth.Workload("dec_det", H=4, G=16, seqs=[(1, 20000), (1, 3333)], seed=9)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    o1, s1, n1 = run_forward(w, x, dx=dx)
    o2, s2, n2 = run_forward(w, x, dx=dx)
    assert torch.equal(s1, s2) and torch.equal(n1, n2)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("name", ["decode_1x4096", "decode_4x65536", "decode_1x262144"])
def test_decode_workloads_full_size(name):
    w = synth.workload(name)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_decode_max_cache_len():
    """The largest supported cache (2^21 tokens, 32,768 blocks): the selection
    reads its pooled scores in rounds from memory (beyond the register and
    shared-memory paths)."""
    w = synth.Workload("dec_max_len", H=1, G=16, seqs=[(1, 1 << 21), (1, 70000)], seed=31)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_decode_max_num_seqs():
    """4,096 decode sequences (the supported maximum) with ragged short caches:
    the scan's prefix sum over sequences runs in several chunks and the
    attention grid is 4,096 deep."""
    lens = synth.ragged_lengths(5, 4096, 1, 400)
    w = synth.Workload("dec_many", H=2, G=4, seqs=[(1, L) for L in lens], seed=32)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_decode_family_max_rows_many_sequences():
    """4,096 sequences of 8 drafted rows each: 32,768 attention grid rows."""
    lens = synth.ragged_lengths(6, 4096, 8, 200)
    w = synth.Workload("dec_many_rows", H=1, G=2, seqs=[(8, L) for L in lens], seed=33)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)
