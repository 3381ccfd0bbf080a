"""Inconsistent device metadata on the GPU: kernels clamp, set the workspace
error word (bit 2, bad metadata) and never read or write outside the stated
extents; the context stays usable (a clean call afterwards is exact)."""
import pytest
import torch

import synth
from gpu_common import (assert_out_close, assert_selection_equal, device_inputs, msa, oracle_forward, problem,
                        run_forward)

pytestmark = pytest.mark.gpu

BAD_METADATA = 2


def forward_with(w, x, mutate):
    m = msa()
    dx = device_inputs(x)
    pb = problem(w, x)
    mutate(pb)
    ws = pb.workspace()
    m.forward(pb, dx["q"], dx["iq"], dx["k"], dx["v"], dx["ik"], workspace=ws)
    torch.cuda.synchronize()
    return m.error_word(ws)


@pytest.mark.parametrize("seqs", [[(1, 3000), (1, 500)], [(100, 3000), (50, 500)], [(1, 3000), (60, 500)]])
@pytest.mark.parametrize("bad", ["len_zero", "len_past_bound"])
def test_bad_cache_len_flagged(seqs, bad):
    w = synth.Workload("err_len", H=2, G=16, seqs=seqs, seed=81)
    x = synth.make_inputs(w)

    def mutate(pb):
        pb.cache_lens[1] = 0 if bad == "len_zero" else pb.max_cache_len + 64

    assert forward_with(w, x, mutate) & BAD_METADATA
    # the context is intact: a clean call is still exact
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_cache_start_past_the_cache_flagged():
    w = synth.Workload("err_start", H=2, G=16, seqs=[(1, 3000), (70, 500)], seed=82)
    x = synth.make_inputs(w)

    def mutate(pb):
        pb.cache_starts[1] = pb.cache_tokens  # the sequence would run past the cache

    assert forward_with(w, x, mutate) & BAD_METADATA


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_given_selection_outside_causal_range_flagged(kind):
    m = msa()
    seqs = [(1, 2000), (1, 300)] if kind == "decode" else [(20, 2000), (30, 300)]
    w = synth.Workload("err_sel", H=2, G=16, seqs=seqs, seed=83)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    ref = oracle_forward(w, x)
    sel = torch.from_numpy(ref["sel"]).cuda()
    nsel = torch.from_numpy(ref["nsel"]).cuda()
    sel[-1, 0, 0] = 10_000  # a block far past the row's position
    ws = pb.workspace()
    fn = m.attend_decode if kind == "decode" else m.attend_prefill
    fn(pb, dx["q"], dx["k"], dx["v"], sel, nsel, workspace=ws)
    torch.cuda.synchronize()
    assert m.error_word(ws) & BAD_METADATA


@pytest.mark.parametrize("seqs,claimed", [([(1, 3000), (3, 2000)], 1), ([(1, 3000), (3, 2000), (1, 1500)], 2)])
def test_rows_beyond_max_rows_per_seq_flagged(seqs, claimed):
    """max_rows_per_seq understated: a decode-family sequence has more rows than
    the pooled scores give each sequence slots for (min(max_rows_per_seq, 8)).
    The scan skips that sequence (no write into the next sequence's slots or
    past the buffer) and the attention sets the error word; a clean call
    afterwards is exact."""
    w = synth.Workload("err_rows", H=2, G=16, seqs=seqs, seed=84)
    x = synth.make_inputs(w)

    def mutate(pb):
        pb.c.max_rows_per_seq = claimed

    assert forward_with(w, x, mutate) & BAD_METADATA
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    """A barrier wait that nothing completes gives up after its limit, sets the
    timeout bit of the error word and returns; the next call is exact."""
    m = msa()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    m.check_wait_timeout(ws, limit_us=20000)
    torch.cuda.synchronize()
    assert m.error_word(ws) & m.ERR_WAIT_TIMEOUT
    w = synth.Workload("after_timeout", H=2, G=16, seqs=[(1, 3000), (40, 900)], seed=81)
    x = synth.make_inputs(w)
    out, sel, nsel = run_forward(w, x)
    ref = oracle_forward(w, x)
    assert_selection_equal(sel, nsel, ref)
    assert_out_close(out, ref["out"], torch.float32)
