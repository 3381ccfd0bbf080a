"""Decode family with several rows per sequence (1 to 8: drafted windows):
one index-key pass serves all of a sequence's rows, each row with its own
causal position, selection and attention.  GPU against the oracle:
selections bit-exact, outputs within tolerance; the boundary to the
prompt-chunk kernels (9 rows); the staged decode attention; paged caches."""
import numpy as np
import pytest
import torch

import synth
from gpu_common import (assert_out_close, assert_selection_equal, device_inputs, msa, oracle_forward, problem,
                        run_forward, to_dev)

pytestmark = pytest.mark.gpu

SEQS = [(2, 5000), (3, 64), (4, 65), (5, 1000), (8, 4097), (1, 777), (7, 8), (6, 129)]


@pytest.mark.parametrize("H,G", [(1, 16), (4, 16), (8, 2), (2, 13)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_multirow_forward(H, G, out_dtype):
    w = synth.Workload("multirow", H=H, G=G, seqs=SEQS, seed=50 + H * 3 + G)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x, out_dtype)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], out_dtype)


@pytest.mark.parametrize("hint", ["auto", -1])
def test_multirow_boundary_with_prompt_chunks(hint):
    """8 rows take the decode kernels, 9 the prompt-chunk kernels, in one call."""
    w = synth.Workload("multirow_edge", H=4, G=16, seqs=[(8, 3000), (9, 3000), (1, 2000), (200, 1300)], seed=61)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x, num_decode_seqs=hint)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_multirow_attend_decode_given_selection():
    m = msa()
    w = synth.Workload("multirow_given", H=4, G=16, seqs=[(4, 2500), (2, 700), (8, 9000)], seed=62)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    ref = oracle_forward(w, x)
    out = m.attend_decode(pb, dx["q"], dx["k"], dx["v"], torch.from_numpy(ref["sel"]).cuda(),
                          torch.from_numpy(ref["nsel"]).cuda())
    torch.cuda.synchronize()
    assert_out_close(out, ref["out"], torch.float32)


def test_multirow_paged():
    m = msa()
    w = synth.Workload("multirow_paged", H=4, G=16, seqs=[(4, 6000), (3, 100), (8, 2049)], seed=63)
    x = synth.make_inputs(w)
    pl = synth.paged_layout(w, x, 256, seed=9)
    pb = m.Problem(w.H, w.G, w.seqs, "cuda", top_k=w.top_k, scale=w.softmax_scale,
                   block_table=torch.from_numpy(pl["table"]), page_size=256, cache_tokens=pl["num_pages"] * 256)
    d = {k: to_dev(x[k]) for k in ("q", "iq")}
    d.update({k: to_dev(pl[k]) for k in ("k", "v", "ik")})
    ws = pb.workspace()
    out, sel, nsel = m.forward(pb, d["q"], d["iq"], d["k"], d["v"], d["ik"], workspace=ws)
    torch.cuda.synchronize()
    assert m.error_word(ws) == 0
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_multirow_4x4_at_65536():
    """Four sequences with four drafted rows each over 65,536 cached tokens."""
    w = synth.Workload("decode_4x4_65536", H=4, G=16, seqs=[(4, 65536)] * 4, seed=64)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    err = assert_out_close(out, ref["out"], torch.float32)
    assert np.isfinite(err)


@pytest.mark.parametrize("count", ["auto", 0, "over", "under"])
def test_mixed_batch_decode_row_count(count):
    """The host's count of decode-family rows sizes the decode attention's grid
    in a mixed batch: exact ('auto'), unknown (0: one entry per row slot) or
    above the device metadata's count give the oracle's outputs; a count below
    it sets the bad-metadata bit."""
    m = msa()
    w = synth.Workload("mixed_rows", H=4, G=16, seqs=[(3, 3000), (200, 1300), (1, 2000), (8, 900), (64, 700)],
                       seed=64)
    x = synth.make_inputs(w)
    exact = 3 + 1 + 8
    n = {"auto": "auto", 0: 0, "over": exact + 5, "under": exact - 2}[count]
    dx = device_inputs(x)
    pb = problem(w, x, num_decode_rows=n)
    ws = pb.workspace()
    out, sel, nsel = m.forward(pb, dx["q"], dx["iq"], dx["k"], dx["v"], dx["ik"], workspace=ws)
    torch.cuda.synchronize()
    if count == "under":
        assert m.error_word(ws) & m.ERR_BAD_METADATA
        return
    assert m.error_word(ws) == 0
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)
