"""The allocation-free decode attention entry point.

msa_attend_decode_noalloc serves callers that cannot call cudaMalloc (for
example code enqueued inside a framework's CUDA-graph capture that forbids
allocation, or a plug-in that does not own its process's allocator): it
takes no workspace and keeps its scratch in a fixed device array inside the
library.  These tests call it through the C ABI and check it against the
workspace-based msa_attend_decode and against the fp64 oracle on the same
inputs, twice in a row (the shared scratch keeps the previous call's
contents).  The file is named so that pytest collects it last."""
import ctypes as C

import numpy as np
import pytest
import torch

import synth
from gpu_common import TOL_F32, device_inputs, msa, oracle_forward, problem


def _noalloc(m, pb, dx, sel, nsel, out):
    return m.lib().msa_attend_decode_noalloc(C.byref(pb.c), C.c_void_p(dx["q"].data_ptr()),
                                             C.c_void_p(dx["k"].data_ptr()), C.c_void_p(dx["v"].data_ptr()),
                                             C.c_void_p(sel.data_ptr()), C.c_void_p(nsel.data_ptr()),
                                             C.c_void_p(out.data_ptr()),
                                             C.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    m = msa()
    w = synth.Workload("noalloc", H=4, G=16, seqs=[(1, L) for L in [70, 4000, 65, 12345, 1, 2048, 999, 30000]],
                       seed=77)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    ref = oracle_forward(w, x)
    sel = torch.from_numpy(ref["sel"]).cuda()
    nsel = torch.from_numpy(ref["nsel"]).cuda()
    expected = m.attend_decode(pb, dx["q"], dx["k"], dx["v"], sel, nsel)
    torch.cuda.synchronize()
    exp = expected.cpu().numpy()
    assert np.abs(exp - ref["out"]).max() <= TOL_F32
    for _ in range(2):
        out = torch.full_like(expected, float("nan"))
        st = _noalloc(m, pb, dx, sel, nsel, out)
        assert st == 0, m.lib().msa_last_error()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        assert np.abs(got - exp).max() <= TOL_F32  # the workspace entry point
        assert np.abs(got - ref["out"]).max() <= TOL_F32  # the fp64 oracle


@pytest.mark.gpu
def test_noalloc_empty_selection_writes_zeros_like_workspace_entry_point():
    """A given count of kept blocks below 1 (an empty softmax) gives zero
    outputs for that (row, KV head) from both entry points; the other
    (row, head) pairs keep their oracle values."""
    m = msa()
    w = synth.Workload("noalloc_empty", H=2, G=16, seqs=[(1, L) for L in [500, 3000, 64]], seed=5)
    x = synth.make_inputs(w)
    dx = device_inputs(x)
    pb = problem(w, x)
    ref = oracle_forward(w, x)
    nsel_np = ref["nsel"].copy()
    nsel_np[1, 0] = 0
    sel = torch.from_numpy(ref["sel"]).cuda()
    nsel = torch.from_numpy(nsel_np).cuda()
    ws = pb.workspace()
    expected = m.attend_decode(pb, dx["q"], dx["k"], dx["v"], sel, nsel, workspace=ws)
    torch.cuda.synchronize()
    assert m.error_word(ws) & m.ERR_BAD_METADATA
    exp = expected.cpu().numpy()
    for _ in range(2):
        out = torch.full_like(expected, float("nan"))
        assert _noalloc(m, pb, dx, sel, nsel, out) == 0, m.lib().msa_last_error()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.array_equal(got[1, 0:16], np.zeros_like(got[1, 0:16]))
        assert np.array_equal(exp[1, 0:16], got[1, 0:16])
        keep = np.ones(got.shape[:2], dtype=bool)
        keep[1, 0:16] = False
        assert np.abs(got[keep] - ref["out"][keep]).max() <= TOL_F32
        assert np.abs(exp[keep] - ref["out"][keep]).max() <= TOL_F32


def test_noalloc_rejects_problems_beyond_its_scratch():
    m = msa()
    pb = m.MsaProblem(num_seqs=9, num_kv_heads=4, group_size=16, head_dim=128, index_dim=64, block_size=64,
                      top_k=16, softmax_scale=0.088, out_dtype=0, total_rows=9, max_rows_per_seq=1,
                      max_cache_len=4096, cache_tokens=9 * 4096, num_decode_seqs=9, cu_rows=256, cache_lens=512,
                      cache_starts=768)
    fake = C.c_void_p(1 << 30)
    st = m.lib().msa_attend_decode_noalloc(C.byref(pb), fake, fake, fake, fake, fake, fake, None)
    assert st == 2  # MSA_ERR_UNSUPPORTED, before anything is enqueued
    assert b"32" in m.lib().msa_last_error()
