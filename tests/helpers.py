"""Shared test helpers: golden fixtures, pinned checks of the CPU oracle.

Each ``check_*`` function pins one part of the oracle to something other than
itself (a hand-worked fixture, a closed form, a library routine, brute force
or an invariant).  They take an optional ``lib_path`` so the planted-mistake
test can run the same checks against deliberately broken oracle builds.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import torch

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def read_cases(name):
    path = os.path.join(ROOT, "tests", "golden", name)
    out = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append([c.strip() for c in line.split("|")])
    return out


def ints(s):
    return [int(v) for v in s.split()]


def bf16_bits(values) -> np.ndarray:
    """bf16 bit patterns of values that bf16 holds exactly (small integers, halves)."""
    f = np.asarray(values, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def to_f64(bits) -> np.ndarray:
    return synth.bf16_to_f32(np.asarray(bits)).astype(np.float64)


# --------------------------------------------------------------------------
# inputs that realise given pooled scores through the full forward
# --------------------------------------------------------------------------

def realize_pooled(m, top_k, S=64, H=1, G=1, D=128, Di=64, seed=7):
    """One decode row whose pooled index scores per block are exactly m.

    iq is the unit vector e_0, so s_t = ik[t, 0]; every position holds -8
    except one per block, which holds m_j.  The row sits 5 positions into
    its local block J = len(m) - 1.
    """
    J = len(m) - 1
    p = S * J + 5
    L = p + 1
    w = synth.Workload("realize", H=H, G=G, seqs=[(1, L)], D=D, Di=Di, S=S, top_k=top_k, seed=seed)
    x = synth.make_inputs(w)
    iq = np.zeros((1, H, Di), dtype=np.float32)
    iq[:, :, 0] = 1.0
    ikv = np.full((L, H, Di), -8.0, dtype=np.float32)
    for j, mj in enumerate(m):
        t = S * j + (j % 6 if j == J else j % S)
        ikv[t, :, 0] = mj
    x["iq"] = bf16_bits(iq)
    x["ik"] = bf16_bits(ikv)
    return w, x


# --------------------------------------------------------------------------
# pinned checks
# --------------------------------------------------------------------------

def check_select_golden(lib_path=None):
    for name, k, m, exp in read_cases("select_cases.txt"):
        sel, n = oracle.select(np.array(ints(m), dtype=np.float64), int(k), lib_path=lib_path)
        assert list(sel[:n]) == ints(exp), (name, list(sel[:n]), ints(exp))
        assert all(v == -1 for v in sel[n:]), name


def check_select_golden_through_forward(lib_path=None):
    for name, k, m, exp in read_cases("select_cases.txt"):
        w, x = realize_pooled(ints(m), int(k))
        pr = oracle.Problem.from_workload(w, x)
        r = oracle.forward(pr, x, with_out=False, lib_path=lib_path)
        n = int(r["nsel"][0, 0])
        assert list(r["sel"][0, 0, :n]) == ints(exp), (name, list(r["sel"][0, 0, :n]))


def check_pool_golden(lib_path=None):
    for name, S, s, exp in read_cases("pool_cases.txt"):
        m = oracle.pool(np.array(ints(s), dtype=np.float64), int(S), lib_path=lib_path)
        assert list(m) == ints(exp), (name, list(m))


def check_scores_unit_query(lib_path=None):
    """iq = e_d  =>  s_t = ik[t, h, d] exactly."""
    w = synth.Workload("unit", H=2, G=1, seqs=[(3, 200)], seed=3)
    x = synth.make_inputs(w, with_kv=False)
    pr = oracle.Problem.from_workload(w, x)
    for d, h in [(0, 0), (17, 1), (63, 1)]:
        iq = np.zeros((3, 2, 64), dtype=np.float32)
        iq[:, h, d] = 1.0
        s = oracle.index_scores(pr, bf16_bits(iq), x["ik"], 2, h, lib_path=lib_path)
        assert np.array_equal(s, to_f64(x["ik"][:, h, d])), (d, h)


def check_scores_integer_matmul(lib_path=None):
    """Integer-valued inputs: the scores equal numpy's exact int64 matmul."""
    w = synth.Workload("mm", H=3, G=1, seqs=[(2, 130), (1, 77)], seed=11)
    x = synth.make_inputs(w, with_kv=False)
    pr = oracle.Problem.from_workload(w, x)
    iq = to_f64(x["iq"]).astype(np.int64)
    ik = to_f64(x["ik"]).astype(np.int64)
    for r in range(3):
        b, p = pr.position(r)
        start = int(x["cache_starts"][b])
        for h in range(3):
            ref = ik[start:start + p + 1, h, :] @ iq[r, h, :]
            s = oracle.index_scores(pr, x["iq"], x["ik"], r, h, lib_path=lib_path)
            assert np.array_equal(s, ref.astype(np.float64)), (r, h)


def check_shared_key_integer_matmul(lib_path=None):
    """One index key per position shared by every KV head: each head's scores
    equal numpy's exact int64 matmul of the shared keys with its own query."""
    w = synth.Workload("mm_shared", H=4, G=1, seqs=[(2, 130), (1, 77)], seed=12, ik_heads=1)
    x = synth.make_inputs(w, with_kv=False)
    assert x["ik"].shape[1] == 1
    pr = oracle.Problem.from_workload(w, x)
    iq = to_f64(x["iq"]).astype(np.int64)
    ik = to_f64(x["ik"]).astype(np.int64)
    for r in range(3):
        b, p = pr.position(r)
        start = int(x["cache_starts"][b])
        for h in range(4):
            ref = ik[start:start + p + 1, 0, :] @ iq[r, h, :]
            s = oracle.index_scores(pr, x["iq"], x["ik"], r, h, lib_path=lib_path)
            assert np.array_equal(s, ref.astype(np.float64)), (r, h)


def check_shared_key_equals_replicated(lib_path=None):
    """A shared index key gives exactly the per-head result with that key
    copied into every head."""
    w = synth.Workload("shared_rep", H=3, G=2, seqs=[(1, 2000), (5, 700)], seed=13, ik_heads=1, top_k=6)
    x = synth.make_inputs(w)
    ref = oracle.forward(oracle.Problem.from_workload(w, x), x, lib_path=lib_path)
    x_rep = dict(x)
    x_rep["ik"] = np.ascontiguousarray(np.repeat(x["ik"], w.H, axis=1))
    rep = oracle.forward(oracle.Problem.from_workload(w, x_rep), x_rep, lib_path=lib_path)
    assert np.array_equal(ref["sel"], rep["sel"]) and np.array_equal(ref["nsel"], rep["nsel"])
    assert np.array_equal(ref["out"], rep["out"])


def _dense_reference(w, x, r, h):
    """Dense causal attention of row r, KV head h, over all keys t <= p, by
    torch's scaled_dot_product_attention in float64 (math path on CPU)."""
    pr = oracle.Problem.from_workload(w, x)
    b, p = pr.position(r)
    s0 = int(x["cache_starts"][b])
    q = torch.from_numpy(to_f64(x["q"][r, h * w.G:(h + 1) * w.G, :]))[None]  # [1, G, D]
    k = torch.from_numpy(to_f64(x["k"][s0:s0 + p + 1, h, :]))[None, None].expand(1, w.G, -1, -1)
    v = torch.from_numpy(to_f64(x["v"][s0:s0 + p + 1, h, :]))[None, None].expand(1, w.G, -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(q[:, :, None, :], k, v, scale=w.softmax_scale)
    return o[0, :, 0, :].numpy()


def check_dense_special_case(lib_path=None):
    """Every causal block kept (J < top_k): MSA is dense causal attention."""
    w = synth.Workload("dense", H=2, G=4, seqs=[(1, 1), (70, 900), (1, 1024), (3, 65)], seed=5)
    x = synth.make_inputs(w)
    pr = oracle.Problem.from_workload(w, x)
    rows = [0, 1, 35, 70, 71, 72, 74]
    res = oracle.forward(pr, x, rows=rows, lib_path=lib_path)
    for i, r in enumerate(rows):
        _, p = pr.position(r)
        for h in range(2):
            assert res["nsel"][i, h] == p // 64 + 1
            ref = _dense_reference(w, x, r, h)
            got = res["out"][i, h * 4:(h + 1) * 4]
            assert np.max(np.abs(got - ref)) < 1e-12, (r, h, np.max(np.abs(got - ref)))


def check_explicit_selection(lib_path=None):
    """Attention over a hand-chosen block list equals dense attention over the
    gathered keys of those blocks (positions <= p only)."""
    w = synth.Workload("explicit", H=2, G=3, seqs=[(40, 1500)], seed=9)
    x = synth.make_inputs(w)
    pr = oracle.Problem.from_workload(w, x)
    for r, blocks in [(0, [0, 3, 7, 22]), (39, [1, 2, 23]), (20, [5, 22])]:
        b, p = pr.position(r)
        keys = [t for j in blocks for t in range(64 * j, 64 * j + 64) if t <= p]
        for h in range(2):
            got = oracle.attend(pr, x["q"], x["k"], x["v"], r, h, blocks, lib_path=lib_path)
            q = torch.from_numpy(to_f64(x["q"][r, h * 3:(h + 1) * 3, :]))[:, None, :]
            k = torch.from_numpy(to_f64(x["k"][keys, h, :]))[None].expand(3, -1, -1)
            v = torch.from_numpy(to_f64(x["v"][keys, h, :]))[None].expand(3, -1, -1)
            ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=w.softmax_scale)[:, 0].numpy()
            assert np.max(np.abs(got - ref)) < 1e-12, (r, h)


def check_two_key_closed_form(lib_path=None):
    """D=2, scale 1: scores (0, 0, 1) give weights (1, 1, e); with v = (1,0),
    (0,1), (2,2) the output is ((1+2e)/(2+e), (1+2e)/(2+e))."""
    cu, lens, starts = np.array([0, 1]), np.array([3]), np.array([0])
    pr = oracle.Problem(1, 1, cu, lens, starts, D=2, Di=2, S=2, top_k=16, scale=1.0)
    q = bf16_bits([[[1.0, 0.0]]])
    k = bf16_bits([[[0.0, 0.0]], [[0.0, 5.0]], [[1.0, 0.0]]])
    v = bf16_bits([[[1.0, 0.0]], [[0.0, 1.0]], [[2.0, 2.0]]])
    got = oracle.attend(pr, q, k, v, 0, 0, [0, 1], lib_path=lib_path)
    e = math.e
    exp = (1 + 2 * e) / (2 + e)
    assert abs(got[0, 0] - exp) < 1e-14 and abs(got[0, 1] - exp) < 1e-14, got


def check_constant_values(lib_path=None):
    """v identical at every key  =>  output equals that v."""
    w = synth.Workload("const", H=1, G=16, seqs=[(5, 3000)], seed=13)
    x = synth.make_inputs(w)
    row = bf16_bits(np.linspace(-4, 4, 128).round() / 2)
    x["v"] = np.broadcast_to(row, x["v"].shape).copy()
    pr = oracle.Problem.from_workload(w, x)
    res = oracle.forward(pr, x, lib_path=lib_path)
    assert np.max(np.abs(res["out"] - to_f64(row)[None, None, :])) < 1e-12


def check_single_key(lib_path=None):
    """A row at position 0 attends to its own key only: output = v_0."""
    w = synth.Workload("single", H=2, G=2, seqs=[(1, 1)], seed=17)
    x = synth.make_inputs(w)
    pr = oracle.Problem.from_workload(w, x)
    res = oracle.forward(pr, x, lib_path=lib_path)
    for h in range(2):
        for g in range(2):
            assert np.array_equal(res["out"][0, h * 2 + g], to_f64(x["v"][0, h]))


def check_zero_scale_is_mean(lib_path=None):
    """scale 0: uniform weights, the output is the mean of v over kept keys."""
    w = synth.Workload("mean", H=1, G=2, seqs=[(1, 2000)], seed=19, scale=0.0, top_k=4)
    x = synth.make_inputs(w)
    pr = oracle.Problem.from_workload(w, x)
    res = oracle.forward(pr, x, lib_path=lib_path)
    sel = [s for s in res["sel"][0, 0] if s >= 0]
    p = 1999
    keys = [t for j in sel for t in range(64 * j, 64 * j + 64) if t <= p]
    ref = to_f64(x["v"][keys, 0, :]).mean(axis=0)
    assert np.max(np.abs(res["out"][0, 0] - ref)) < 1e-12


def _is_top_set(m, chosen, J):
    """chosen (non-local) dominates every other candidate j < J under
    (score descending, index ascending)."""
    rest = [j for j in range(J) if j not in chosen]
    return all((m[c] > m[j]) or (m[c] == m[j] and c < j) for c in chosen for j in rest)


def check_select_bruteforce(lib_path=None):
    """Tiny cases: exactly one (k-1)-subset of blocks j < J dominates the rest;
    the selection must be it plus the local block."""
    rng = np.random.default_rng(123)
    for trial in range(60):
        J = int(rng.integers(0, 9))
        k = int(rng.integers(1, 7))
        m = rng.integers(-2, 3, size=J + 1).astype(np.float64)
        winners = [set(c) for c in itertools.combinations(range(J), min(k - 1, J)) if _is_top_set(m, set(c), J)]
        assert len(winners) == 1
        exp = sorted(winners[0] | {J})
        sel, n = oracle.select(m, k, lib_path=lib_path)
        assert list(sel[:n]) == exp, (m, k, list(sel[:n]), exp)


def check_select_invariants(lib_path=None):
    rng = np.random.default_rng(321)
    for trial in range(200):
        J = int(rng.integers(0, 300))
        k = int(rng.integers(1, 20))
        m = rng.integers(-4, 5, size=J + 1).astype(np.float64)
        sel, n = oracle.select(m, k, lib_path=lib_path)
        chosen = list(sel[:n])
        assert n == min(k, J + 1)
        assert J in chosen
        assert chosen == sorted(set(chosen))
        assert all(0 <= c <= J for c in chosen)
        assert all(v == -1 for v in sel[n:])
        assert _is_top_set(m, set(chosen) - {J}, J)


def check_future_blocks_never_selected(lib_path=None):
    """A prompt chunk: hot index keys late in the cache are in the future of
    the early rows and must not be selected by them."""
    w = synth.Workload("future", H=1, G=1, seqs=[(200, 1100)], seed=23, top_k=4)
    x = synth.make_inputs(w, with_kv=False)
    iq = np.zeros((200, 1, 64), dtype=np.float32)
    iq[:, :, 0] = 1.0
    ikv = np.full((1100, 1, 64), -8.0, dtype=np.float32)
    ikv[1000:, :, 0] = 8.0
    ikv[130, :, 0] = 3.0
    x["iq"], x["ik"] = bf16_bits(iq), bf16_bits(ikv)
    pr = oracle.Problem.from_workload(w, x)
    res = oracle.forward(pr, x, with_out=False, lib_path=lib_path)
    for i in range(200):
        _, p = pr.position(i)
        J = p // 64
        sel = list(res["sel"][i, 0, :res["nsel"][i, 0]])
        hot = [j for j in range(J) if 64 * j + 63 >= 1000]
        exp = sorted(set((hot + [2] + [0, 1, 3])[:3]) | {J}) if hot else sorted({2, 0, 1} | {J})
        assert max(sel) == J and sel == exp, (i, p, sel, exp)


# --------------------------------------------------------------------------
# int8 key/value cache (PR #1388, native Metal family commit: int8 values with
# one scale per position and head; read as value = scale * int8)
# --------------------------------------------------------------------------

def _int8_workload(name, seed, scale=None):
    w = synth.Workload(name, H=2, G=4, seqs=[(1, 700), (9, 1300), (1, 64)], seed=seed, kv_dtype="int8",
                       scale=scale)
    return w, synth.make_inputs(w)


def _as_bf16_cache(a8):
    """The same integers stored as bf16 (exact for |v| <= 256)."""
    return bf16_bits(a8.astype(np.float32))


def check_int8_unit_scales_equal_bf16_integers(lib_path=None):
    """All scales 1: the int8 cache reads the same values as a bf16 cache
    holding the same integers, so the outputs are identical."""
    w, x = _int8_workload("int8_unit", 31)
    ones = np.ones_like(x["k_scale"])
    x8 = dict(x, k_scale=ones, v_scale=ones)
    xb = {k: v for k, v in x.items() if k not in ("k_scale", "v_scale")}
    xb["k"], xb["v"] = _as_bf16_cache(x["k"]), _as_bf16_cache(x["v"])
    r8 = oracle.forward(oracle.Problem.from_workload(w, x8), x8, lib_path=lib_path)
    rb = oracle.forward(oracle.Problem.from_workload(w, xb), xb, lib_path=lib_path)
    assert np.array_equal(r8["sel"], rb["sel"])
    assert np.array_equal(r8["out"], rb["out"])


def check_int8_key_scale_is_softmax_scale(lib_path=None):
    """Every key scale 1/4 (a power of two, so every product is exact) and
    value scales 1: the same as a bf16 cache of the integers with the softmax
    scale divided by 4."""
    w, x = _int8_workload("int8_kscale", 37)
    x8 = dict(x, k_scale=np.full_like(x["k_scale"], 0.25), v_scale=np.ones_like(x["v_scale"]))
    wb = synth.Workload(w.name, H=w.H, G=w.G, seqs=w.seqs, seed=w.seed, scale=w.softmax_scale * 0.25)
    xb = {k: v for k, v in x.items() if k not in ("k_scale", "v_scale")}
    xb["k"], xb["v"] = _as_bf16_cache(x["k"]), _as_bf16_cache(x["v"])
    r8 = oracle.forward(oracle.Problem.from_workload(w, x8), x8, lib_path=lib_path)
    rb = oracle.forward(oracle.Problem.from_workload(wb, xb), xb, lib_path=lib_path)
    assert np.max(np.abs(r8["out"] - rb["out"])) < 1e-13


def check_int8_value_scales_closed_form(lib_path=None):
    """Two keys with zero key vectors (equal scores): the output is the mean
    of the two dequantised values, each with its own position's and head's
    scale: (vs_0 * v8_0 + vs_1 * v8_1) / 2."""
    cu, lens, starts = np.array([0, 1]), np.array([2]), np.array([0])
    vs = np.array([[0.5, 3.0], [0.125, 7.0]], dtype=np.float32)  # [position, head]
    pr = oracle.Problem(2, 1, cu, lens, starts, D=2, Di=2, S=2, top_k=16, scale=1.0,
                        k_scale=np.ones((2, 2), dtype=np.float32), v_scale=vs)
    q = bf16_bits([[[1.0, 2.0], [3.0, -1.0]]])
    k = np.zeros((2, 2, 2), dtype=np.int8)
    v = np.array([[[10, -3], [4, 5]], [[-8, 100], [-127, 1]]], dtype=np.int8)
    for h in range(2):
        got = oracle.attend(pr, q, k, v, 0, h, [0], lib_path=lib_path)
        exp = (float(vs[0, h]) * v[0, h].astype(np.float64) + float(vs[1, h]) * v[1, h].astype(np.float64)) / 2
        assert np.max(np.abs(got[0] - exp)) < 1e-15, (h, got, exp)


def check_int8_key_scales_closed_form(lib_path=None):
    """Two keys with the same int8 vector but different scales: scores
    scale * ks_t * (q . k8), so the weights are exp(ks_0 c) and exp(ks_1 c)
    with c = q . k8 = 3; the output weighs the two values by them."""
    cu, lens, starts = np.array([0, 1]), np.array([2]), np.array([0])
    ks = np.array([[0.25], [0.5]], dtype=np.float32)
    pr = oracle.Problem(1, 1, cu, lens, starts, D=2, Di=2, S=2, top_k=16, scale=1.0,
                        k_scale=ks, v_scale=np.ones((2, 1), dtype=np.float32))
    q = bf16_bits([[[1.0, 1.0]]])
    k = np.array([[[1, 2]], [[1, 2]]], dtype=np.int8)
    v = np.array([[[1, 0]], [[0, 1]]], dtype=np.int8)
    got = oracle.attend(pr, q, k, v, 0, 0, [0], lib_path=lib_path)
    w0, w1 = math.exp(0.25 * 3), math.exp(0.5 * 3)
    exp = np.array([w0, w1]) / (w0 + w1)
    assert np.max(np.abs(got[0] - exp)) < 1e-14, (got, exp)


def check_int8_dense_special_case(lib_path=None):
    """Every causal block kept: the int8 cache's MSA output is dense causal
    attention (torch float64 SDPA) over the dequantised keys and values."""
    w, x = _int8_workload("int8_dense", 41)
    pr = oracle.Problem.from_workload(w, x)
    rows = [0, 1, 5, 9, 10]
    res = oracle.forward(pr, x, rows=rows, lib_path=lib_path)
    for i, r in enumerate(rows):
        b, p = pr.position(r)
        if p // 64 + 1 > w.top_k:
            continue
        s0 = int(x["cache_starts"][b])
        for h in range(w.H):
            kd = x["k"][s0:s0 + p + 1, h, :].astype(np.float64) * x["k_scale"][s0:s0 + p + 1, h, None]
            vd = x["v"][s0:s0 + p + 1, h, :].astype(np.float64) * x["v_scale"][s0:s0 + p + 1, h, None]
            qg = torch.from_numpy(to_f64(x["q"][r, h * w.G:(h + 1) * w.G, :]))[None, :, None, :]
            kk = torch.from_numpy(kd)[None, None].expand(1, w.G, -1, -1)
            vv = torch.from_numpy(vd)[None, None].expand(1, w.G, -1, -1)
            ref = torch.nn.functional.scaled_dot_product_attention(qg, kk, vv, scale=w.softmax_scale)[0, :, 0, :]
            got = res["out"][i, h * w.G:(h + 1) * w.G]
            assert np.max(np.abs(got - ref.numpy())) < 1e-12, (r, h)


ALL_CHECKS = [
    check_select_golden, check_select_golden_through_forward, check_pool_golden, check_scores_unit_query,
    check_scores_integer_matmul, check_dense_special_case, check_explicit_selection, check_two_key_closed_form,
    check_constant_values, check_single_key, check_zero_scale_is_mean, check_select_bruteforce,
    check_select_invariants, check_future_blocks_never_selected, check_shared_key_integer_matmul,
    check_shared_key_equals_replicated, check_int8_unit_scales_equal_bf16_integers,
    check_int8_key_scale_is_softmax_scale, check_int8_value_scales_closed_form, check_int8_key_scales_closed_form,
    check_int8_dense_special_case,
]
