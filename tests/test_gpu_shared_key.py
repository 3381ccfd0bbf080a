"""One index key per position shared by every KV head (index_key_heads = 1,
ik [T, 1, Di]): each head's index query meets the same key.  GPU against
the oracle: index scores exact, selections bit-exact, outputs within
tolerance, on every path (decode, drafted windows, prompt chunks, mixed,
paged, staged)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import (assert_out_close, assert_selection_equal, device_inputs, msa, oracle_forward, problem,
                        run_forward, to_dev)

pytestmark = pytest.mark.gpu

SEQS = {
    "decode": [(1, L) for L in [1, 64, 65, 1000, 4097, 9000]],
    "multirow": [(4, 3000), (8, 129), (2, 64)],
    "prefill": [(130, 700), (129, 4000), (64, 64)],
    "mixed": [(1, 3000), (40, 1200), (3, 65), (257, 3100)],
}


@pytest.mark.parametrize("H,G", [(2, 16), (4, 16), (8, 4)])
@pytest.mark.parametrize("kind", ["decode", "multirow", "prefill", "mixed"])
def test_shared_key_forward(kind, H, G):
    w = synth.Workload(f"shared_{kind}", H=H, G=G, seqs=SEQS[kind], seed=70 + H, ik_heads=1)
    x = synth.make_inputs(w)
    assert x["ik"].shape[1] == 1
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_shared_key_staged():
    m = msa()
    w = synth.Workload("shared_staged", H=4, G=16, seqs=[(1, 65), (1, 2000), (3, 777)], seed=71, ik_heads=1)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    scores = m.index_scores(pb, dx["iq"], dx["ik"])
    pr = oracle.Problem.from_workload(w, x)
    sc = scores.cpu().numpy()
    for r in range(pb.total_rows):
        for h in range(w.H):
            ref_s = oracle.index_scores(pr, x["iq"], x["ik"], r, h)
            assert np.array_equal(sc[r, h, :len(ref_s)], ref_s.astype(np.float32))
    sel, nsel = m.select_blocks(pb, scores)
    assert_selection_equal(sel, nsel, oracle_forward(w, x))


def test_shared_key_paged():
    m = msa()
    w = synth.Workload("shared_paged", H=4, G=16, seqs=[(1, 5000), (200, 1300), (4, 700)], seed=72, ik_heads=1)
    x = synth.make_inputs(w)
    pl = synth.paged_layout(w, x, 128, seed=4)
    pb = m.Problem(w.H, w.G, w.seqs, "cuda", top_k=w.top_k, scale=w.softmax_scale, ik_heads=1,
                   block_table=torch.from_numpy(pl["table"]), page_size=128, cache_tokens=pl["num_pages"] * 128)
    d = {k: to_dev(x[k]) for k in ("q", "iq")}
    d.update({k: to_dev(pl[k]) for k in ("k", "v", "ik")})
    ws = pb.workspace()
    out, sel, nsel = m.forward(pb, d["q"], d["iq"], d["k"], d["v"], d["ik"], workspace=ws)
    torch.cuda.synchronize()
    assert m.error_word(ws) == 0
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_shared_key_decode_4x65536():
    w = synth.workload("decode_4x65536_shared_ik")
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)
