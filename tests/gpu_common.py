"""Helpers for the GPU parity tests: move seeded inputs to the device, run
the CUDA path through the C ABI, run the oracle on the same bytes, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

# Tolerances: fp32 output max |err| <= 2e-3, bf16 output <= 1.6e-2, against
# the fp64 oracle; selections bit-exact.
TOL_F32 = 2e-3
TOL_BF16 = 1.6e-2


def msa():
    import block_sparse_attention_index_gb300 as m  # noqa: E402  (needs the built library)
    return m


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 device tensor (same bytes)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def device_inputs(x: dict, device="cuda") -> dict:
    d = {k: to_dev(x[k], device) for k in ("q", "iq", "ik")}
    if "k" in x:
        for k in ("k", "v"):
            # int8 caches go as they are; bf16 bit patterns as bf16
            d[k] = torch.from_numpy(np.ascontiguousarray(x[k])).to(device) if x[k].dtype == np.int8 \
                else to_dev(x[k], device)
    for k in ("k_scale", "v_scale"):
        if k in x:
            d[k] = torch.from_numpy(np.ascontiguousarray(x[k])).to(device)
    return d


def problem(w: synth.Workload, x: dict, out_dtype=torch.float32, device="cuda", **kw):
    m = msa()
    if "k_scale" in x and "k_scale" not in kw:  # an int8 key/value cache
        kw = dict(kw, k_scale=torch.from_numpy(x["k_scale"]), v_scale=torch.from_numpy(x["v_scale"]))
    return m.Problem(w.H, w.G, w.seqs, device, top_k=w.top_k, scale=w.softmax_scale, out_dtype=out_dtype,
                     cache_starts=[int(s) for s in x["cache_starts"]], cache_tokens=int(sum(L for _, L in w.seqs)),
                     ik_heads=w.ik_heads, **kw)


def run_forward(w, x, out_dtype=torch.float32, dx=None, **kw):
    m = msa()
    dx = dx or device_inputs(x)
    pb = problem(w, x, out_dtype, **kw)
    ws = pb.workspace()
    out, sel, nsel = m.forward(pb, dx["q"], dx["iq"], dx["k"], dx["v"], dx["ik"], workspace=ws)
    torch.cuda.synchronize()
    assert m.error_word(ws) == 0
    return out, sel, nsel


def oracle_forward(w, x, rows=None, with_out=True):
    pr = oracle.Problem.from_workload(w, x)
    return oracle.forward(pr, x, rows=rows, with_out=with_out)


def assert_selection_equal(sel_gpu, nsel_gpu, ref, rows=None):
    sg = sel_gpu.cpu().numpy()
    ng = nsel_gpu.cpu().numpy()
    if rows is not None:
        sg, ng = sg[rows], ng[rows]
    bad = np.argwhere((sg != ref["sel"]).any(axis=2) | (ng != ref["nsel"]))
    assert len(bad) == 0, f"{len(bad)} (row, head) selections differ; first {bad[:3].tolist()}: " \
                          f"gpu {sg[tuple(bad[0])].tolist()} vs oracle {ref['sel'][tuple(bad[0])].tolist()}"


def assert_out_close(out_gpu, ref_out, out_dtype, rows=None):
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        o = o[rows]
    err = np.abs(o - ref_out)
    tol = TOL_BF16 if out_dtype == torch.bfloat16 else TOL_F32
    assert np.isfinite(o).all(), "non-finite output"
    assert err.max() <= tol, f"max |err| {err.max():.3g} > {tol} at {np.unravel_index(err.argmax(), err.shape)}"
    return float(err.max())
