"""int8 key/value cache (PR #1388, native Metal family commit: keys and
values cached as int8 with one scale per position and head): the CUDA path
against the oracle's reading k = k_scale * k8, v = v_scale * v8 on the same
seeded bytes.  Selections bit-exact (they use only the bf16 index keys),
outputs within the fp32 / bf16 tolerances."""
import numpy as np
import pytest
import torch

import synth
from gpu_common import (assert_out_close, assert_selection_equal, device_inputs, msa, oracle_forward, problem,
                        run_forward)

pytestmark = pytest.mark.gpu

DECODE_SEQS = [(1, 1), (1, 63), (1, 64), (1, 65), (1, 1023), (1, 1025), (1, 4096), (1, 20000)]


def _w(name, seqs, H=4, G=16, seed=0, **kw):
    return synth.Workload(name, H=H, G=G, seqs=seqs, seed=seed, kv_dtype="int8", **kw)


@pytest.mark.parametrize("H,G", [(1, 16), (4, 16), (8, 2), (2, 13)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_int8_decode_forward(H, G, out_dtype):
    w = _w("int8_decode", DECODE_SEQS, H=H, G=G, seed=70 + H + G)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x, out_dtype)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], out_dtype)


def test_int8_drafted_windows():
    """Several decode rows per sequence (1 to 8) from an int8 cache."""
    w = _w("int8_multirow", [(2, 5000), (3, 64), (8, 4097), (1, 777), (7, 8), (5, 1300)], seed=81)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_int8_attend_decode_given_selection():
    m = msa()
    w = _w("int8_given", [(1, 3000), (4, 700), (1, 9000)], seed=82)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    ref = oracle_forward(w, x)
    out = m.attend_decode(pb, dx["q"], dx["k"], dx["v"], torch.from_numpy(ref["sel"]).cuda(),
                          torch.from_numpy(ref["nsel"]).cuda())
    torch.cuda.synchronize()
    assert_out_close(out, ref["out"], torch.float32)


def test_int8_extreme_values_and_scales():
    """Values at both ends of int8 (-128 and 127) and scales spanning 2^-20 to
    2^6: the widening to bf16 and the scale factors stay exact enough."""
    w = _w("int8_extreme", [(1, 2000), (2, 700)], seed=83)
    x = synth.make_inputs(w)
    rng = np.random.default_rng(83)
    for k in ("k", "v"):
        a = x[k]
        a[::3] = -128
        a[1::5] = 127
    x["k_scale"] = (2.0 ** rng.integers(-8, -3, size=x["k_scale"].shape)).astype(np.float32)
    x["v_scale"] = (2.0 ** rng.integers(-20, 7, size=x["v_scale"].shape)).astype(np.float32)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    o = out.cpu().numpy().astype(np.float64)
    scale = np.maximum(1.0, np.abs(ref["out"]).max(axis=2, keepdims=True))
    assert np.isfinite(o).all()
    assert (np.abs(o - ref["out"]) / scale).max() <= 2e-3


def test_int8_paged_decode():
    m = msa()
    w = _w("int8_paged", [(1, 6000), (3, 100), (8, 2049), (1, 64)], seed=84)
    x = synth.make_inputs(w)
    pl = synth.paged_layout(w, x, 128, seed=11)
    pb = m.Problem(w.H, w.G, w.seqs, "cuda", top_k=w.top_k, scale=w.softmax_scale,
                   block_table=torch.from_numpy(pl["table"]), page_size=128, cache_tokens=pl["num_pages"] * 128,
                   k_scale=torch.from_numpy(pl["k_scale"]), v_scale=torch.from_numpy(pl["v_scale"]))
    dev = {k: torch.from_numpy(np.ascontiguousarray(pl[k])).cuda() for k in ("k", "v")}
    dq = device_inputs({k: x[k] for k in ("q", "iq")} | {"ik": pl["ik"]})
    ws = pb.workspace()
    out, sel, nsel = m.forward(pb, dq["q"], dq["iq"], dev["k"], dev["v"], dq["ik"], workspace=ws)
    torch.cuda.synchronize()
    assert m.error_word(ws) == 0
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_int8_decode_4x65536_full_size():
    """The headline decode workload with an int8 cache, every row checked."""
    w = synth.workload("decode_4x65536_int8")
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_int8_not_taken_by_allocation_free_entry_point():
    m = msa()
    w = _w("int8_noalloc", [(1, 500)], seed=85)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    sel, nsel = pb.new_sel()
    with pytest.raises(m.MsaError) as e:
        m.attend_decode_noalloc(pb, dx["q"], dx["k"], dx["v"], sel, nsel)
    assert e.value.status == 2  # MSA_ERR_UNSUPPORTED


PROMPT_SEQS = [(200, 1300), (65, 65), (130, 5000), (9, 3000), (1, 2000)]


@pytest.mark.parametrize("H,G", [(1, 16), (4, 16), (2, 13), (8, 8)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_int8_prompt_chunks(H, G, out_dtype):
    """Prompt chunks (and a decode row beside them) from an int8 cache: the
    tcgen05 attention widens the int8 tiles to bf16 in shared memory."""
    w = _w("int8_prompt", PROMPT_SEQS, H=H, G=G, seed=90 + H + G)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x, out_dtype)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], out_dtype)


def test_int8_prompt_extreme_values_and_scales():
    """The same extremes for prompt chunks (the tcgen05 attention): value
    scales from 2^-20 to 2^6 in the same blocks, so P (weight x value scale)
    needs bf16's exponent range for the keys with small scales to keep their
    share."""
    w = _w("int8_prompt_extreme", [(300, 2000), (70, 900)], seed=87)
    x = synth.make_inputs(w)
    rng = np.random.default_rng(87)
    for k in ("k", "v"):
        a = x[k]
        a[::3] = -128
        a[1::5] = 127
    x["k_scale"] = (2.0 ** rng.integers(-8, -3, size=x["k_scale"].shape)).astype(np.float32)
    x["v_scale"] = (2.0 ** rng.integers(-20, 7, size=x["v_scale"].shape)).astype(np.float32)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    o = out.cpu().numpy().astype(np.float64)
    scale = np.maximum(1.0, np.abs(ref["out"]).max(axis=2, keepdims=True))
    assert np.isfinite(o).all()
    assert (np.abs(o - ref["out"]) / scale).max() <= 2e-3


def _widen_plan(seqs, only_multi_row, top_k=16, S=64):
    """The library's choice for an int8 prompt-chunk attention: widen the read
    sequences once into the workspace when each widened position serves at
    least four kept key rows on average (host counts exact, as the binding
    fills them)."""
    R = sum(n for n, _ in seqs)
    n = sum(1 for r, _ in seqs if r > 8) if only_multi_row else len(seqs)
    slot_rows = -(-max(L for _, L in seqs) // S) * S
    return n >= 1 and R * top_k * S >= 4 * n * slot_rows


@pytest.mark.parametrize("seqs,widened", [
    ([(200, 1300), (9, 3000), (128, 4096), (1, 2000)], True),  # ragged, whole-block and decode beside
    ([(9, 20000), (1, 3000)], False),                           # few rows over a long prefix
    ([(40, 4000), (3, 700), (12, 129)], True),
])
def test_int8_prompt_widened_once_or_per_item(seqs, widened):
    """Both int8 prompt-chunk forms: the sequences widened once per call into
    the workspace (one more kernel), or the tiles widened by the attention."""
    assert _widen_plan(seqs, True) == widened
    w = _w("int8_prompt_forms", seqs, seed=95 + len(seqs))
    x = synth.make_inputs(w)
    pb = problem(w, x)
    dec = any(n <= 8 for n, _ in seqs)
    assert pb.forward_launches() == (2 if dec else 0) + (3 if widened else 2)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_int8_prompt_widened_decode_count_unknown():
    """num_decode_seqs = -1: the copy has room for every sequence that could
    have more than 8 rows, and the slots go to those that do."""
    seqs = [(1, 3000), (30, 2100), (2, 500), (17, 64)]
    w = _w("int8_prompt_unknown_count", seqs, seed=97)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x, num_decode_seqs=-1)
    # widened: 50 rows x 16 x 64 kept key rows >= 4 x min(4 sequences, 50 // 9) x 3,008 positions
    assert pb.forward_launches() == 5
    ws = pb.workspace()
    out, sel, nsel = msa().forward(pb, dx["q"], dx["iq"], dx["k"], dx["v"], dx["ik"], workspace=ws)
    torch.cuda.synchronize()
    assert msa().error_word(ws) == 0
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_int8_prompt_widened_many_sequences():
    """More than 256 sequences (the widening pass's slot prefix gives each
    thread several), prompt chunks of 9 to 12 rows interleaved with decode
    rows that are not widened, ragged lengths."""
    rng = np.random.default_rng(96)
    seqs = []
    for i in range(330):
        if i % 5 == 4:
            seqs.append((1, int(rng.integers(1, 300))))
        else:
            L = int(rng.integers(12, 260))
            seqs.append((int(rng.integers(9, 13)), L))
    assert _widen_plan(seqs, True)
    w = _w("int8_prompt_many", seqs, H=2, G=4, seed=96)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


@pytest.mark.parametrize("seqs", [[(300, 2500), (17, 700)], [(1, 3000), (4, 700), (1, 9000)]])
def test_int8_attend_prefill_both_forms(seqs):
    """msa_attend_prefill on every sequence of the batch: widened once (many
    rows) or tile by tile (a few rows over long prefixes)."""
    m = msa()
    w = _w("int8_prefill_forms", seqs, seed=93)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    ref = oracle_forward(w, x)
    ws = pb.workspace()
    out = m.attend_prefill(pb, dx["q"], dx["k"], dx["v"], torch.from_numpy(ref["sel"]).cuda(),
                           torch.from_numpy(ref["nsel"]).cuda(), workspace=ws)
    torch.cuda.synchronize()
    assert m.error_word(ws) == 0
    assert_out_close(out, ref["out"], torch.float32)


def test_int8_attend_prefill_given_selection():
    m = msa()
    w = _w("int8_prefill_given", [(300, 2500), (17, 700)], seed=91)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    ref = oracle_forward(w, x)
    out = m.attend_prefill(pb, dx["q"], dx["k"], dx["v"], torch.from_numpy(ref["sel"]).cuda(),
                           torch.from_numpy(ref["nsel"]).cuda())
    torch.cuda.synchronize()
    assert_out_close(out, ref["out"], torch.float32)


@pytest.mark.parametrize("page", [64, 256, 1024])
def test_int8_paged_prompt_chunk(page):
    m = msa()
    w = _w("int8_paged_prompt", [(256, 3000), (1, 900), (40, 200)], seed=92)
    x = synth.make_inputs(w)
    pl = synth.paged_layout(w, x, page, seed=12)
    pb = m.Problem(w.H, w.G, w.seqs, "cuda", top_k=w.top_k, scale=w.softmax_scale,
                   block_table=torch.from_numpy(pl["table"]), page_size=page, cache_tokens=pl["num_pages"] * page,
                   k_scale=torch.from_numpy(pl["k_scale"]), v_scale=torch.from_numpy(pl["v_scale"]))
    dev = {k: torch.from_numpy(np.ascontiguousarray(pl[k])).cuda() for k in ("k", "v")}
    dq = device_inputs({k: x[k] for k in ("q", "iq")} | {"ik": pl["ik"]})
    ws = pb.workspace()
    out, sel, nsel = m.forward(pb, dq["q"], dq["iq"], dev["k"], dev["v"], dq["ik"], workspace=ws)
    torch.cuda.synchronize()
    assert m.error_word(ws) == 0
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_int8_prefill_4096_at_8192_full_size():
    """The 4,096-row prompt chunk at an 8,192-token prefix from an int8 cache."""
    w = synth.workload("prefill_4096_at_8192_int8")
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)
