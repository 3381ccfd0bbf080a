"""Paged caches (a block table per sequence, pages shuffled in a pool whose
unused rows hold other random values) on the GPU, against the oracle run on
the same caches laid out contiguously: selections bit-exact, outputs within
tolerance, index scores exact; every entry point; a page number outside the
pool sets the device error word instead of being read."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import assert_out_close, assert_selection_equal, msa, oracle_forward, to_dev

pytestmark = pytest.mark.gpu

SEQS = {
    "decode": [(1, L) for L in [1, 63, 64, 65, 1000, 4097, 5000]],
    "prefill": [(130, 700), (2, 5), (129, 4000), (64, 64)],
    "mixed": [(1, 3000), (40, 1200), (1, 65), (257, 3100)],
}


def paged_problem(w, pl, out_dtype=torch.float32, **kw):
    return msa().Problem(w.H, w.G, w.seqs, "cuda", top_k=w.top_k, scale=w.softmax_scale, out_dtype=out_dtype,
                         block_table=torch.from_numpy(pl["table"]), page_size=pl["page_size"],
                         cache_tokens=pl["num_pages"] * pl["page_size"], **kw)


def paged_inputs(x, pl):
    d = {k: to_dev(x[k]) for k in ("q", "iq")}
    for k in ("k", "v", "ik"):
        d[k] = to_dev(pl[k])
    return d


def run_paged(w, x, pl, out_dtype=torch.float32):
    m = msa()
    pb = paged_problem(w, pl, out_dtype)
    d = paged_inputs(x, pl)
    ws = pb.workspace()
    out, sel, nsel = m.forward(pb, d["q"], d["iq"], d["k"], d["v"], d["ik"], workspace=ws)
    torch.cuda.synchronize()
    return out, sel, nsel, m.error_word(ws)


@pytest.mark.parametrize("page", [64, 256, 1024])
@pytest.mark.parametrize("kind", ["decode", "prefill", "mixed"])
def test_paged_forward(kind, page):
    w = synth.Workload(f"paged_{kind}", H=4, G=16, seqs=SEQS[kind], seed=40 + page // 64)
    x = synth.make_inputs(w)
    pl = synth.paged_layout(w, x, page, seed=page)
    out, sel, nsel, err = run_paged(w, x, pl)
    assert err == 0
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_paged_forward_bf16_out_h2():
    w = synth.Workload("paged_h2", H=2, G=8, seqs=[(1, 2500), (70, 900), (1, 129)], seed=77)
    x = synth.make_inputs(w)
    pl = synth.paged_layout(w, x, 128, seed=5)
    out, sel, nsel, err = run_paged(w, x, pl, torch.bfloat16)
    assert err == 0
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.bfloat16)


def test_paged_staged_entry_points():
    """msa_index_scores exact, msa_select_blocks bit-exact, both attention
    forms and the allocation-free decode attention on the oracle's selection."""
    m = msa()
    w = synth.Workload("paged_staged", H=4, G=16, seqs=[(1, 65), (1, 2000), (1, 7777)], seed=12)
    x = synth.make_inputs(w)
    pl = synth.paged_layout(w, x, 64, seed=3)
    pb = paged_problem(w, pl)
    d = paged_inputs(x, pl)
    scores = m.index_scores(pb, d["iq"], d["ik"])
    pr = oracle.Problem.from_workload(w, x)
    sc = scores.cpu().numpy()
    for r in range(pb.total_rows):
        for h in range(w.H):
            ref_s = oracle.index_scores(pr, x["iq"], x["ik"], r, h)
            assert np.array_equal(sc[r, h, :len(ref_s)], ref_s.astype(np.float32))
    sel, nsel = m.select_blocks(pb, scores)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    sel_o = torch.from_numpy(ref["sel"]).cuda()
    nsel_o = torch.from_numpy(ref["nsel"]).cuda()
    assert_out_close(m.attend_decode(pb, d["q"], d["k"], d["v"], sel_o, nsel_o), ref["out"], torch.float32)
    assert_out_close(m.attend_decode_noalloc(pb, d["q"], d["k"], d["v"], sel_o, nsel_o), ref["out"], torch.float32)


def test_paged_attend_prefill_given_selection():
    m = msa()
    w = synth.Workload("paged_pre_given", H=4, G=16, seqs=[(100, 3000), (3, 1025)], seed=14)
    x = synth.make_inputs(w)
    pl = synth.paged_layout(w, x, 512, seed=8)
    pb = paged_problem(w, pl)
    d = paged_inputs(x, pl)
    ref = oracle_forward(w, x)
    out = m.attend_prefill(pb, d["q"], d["k"], d["v"], torch.from_numpy(ref["sel"]).cuda(),
                           torch.from_numpy(ref["nsel"]).cuda())
    torch.cuda.synchronize()
    assert_out_close(out, ref["out"], torch.float32)


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_paged_page_outside_pool_sets_error(kind):
    """A page number past the pool is flagged (bad metadata) and never read."""
    w = synth.Workload(f"paged_bad_{kind}", H=2, G=16, seqs=SEQS[kind][:3], seed=2)
    x = synth.make_inputs(w)
    pl = synth.paged_layout(w, x, 64, seed=1)
    pl["table"][0, 0] = pl["num_pages"] + 7
    _, _, _, err = run_paged(w, x, pl)
    assert err & 2


def test_paged_decode_4x65536_full_size():
    """The headline decode workload from a 64-token page pool."""
    w = synth.workload("decode_4x65536")
    x = synth.make_inputs(w)
    pl = synth.paged_layout(w, x, 64, seed=64)
    out, sel, nsel, err = run_paged(w, x, pl)
    assert err == 0
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)
