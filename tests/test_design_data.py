"""Data behind two design choices of the prompt-chunk attention, recomputed on
the CPU (no GPU, no CUDA path).

1. How far neighbouring rows' kept blocks overlap on the 4,096-row chunk at an
   8,192-token prefix (the seeded workload the bar is measured on): the mean
   number of distinct blocks kept by R consecutive rows of one KV head, from
   the oracle's selections.  A tile over the union of R rows' blocks (PR #1388,
   prompt-tile commit: "a tile walks the union of two rows' blocks") issues
   R x union / (R x 16) of the kept FLOPs.
2. How much a single bf16 P (instead of the hi + lo split) costs in accuracy:
   softmax weights rounded to bf16 against fp64, for rows of few keys.

The numbers asserted here are the ones the design notes quote."""
import math

import numpy as np

import oracle
import synth


def union_sizes(sel, R):
    """Mean, min and max number of distinct kept blocks of R consecutive rows,
    over all row groups and KV heads."""
    out = []
    for h in range(sel.shape[1]):
        for r0 in range(0, sel.shape[0], R):
            s = sel[r0:r0 + R, h]
            out.append(len(np.unique(s[s >= 0])))
    out = np.array(out)
    return out.mean(), out.min(), out.max()


def test_selection_overlap_of_consecutive_rows():
    w = synth.workload("prefill_4096_at_8192")
    x = synth.make_inputs(w, with_kv=False)
    ref = oracle.forward(oracle.Problem.from_workload(w, x), x, with_out=False)
    expect = {1: 16.0, 2: 29.56, 4: 52.90, 8: 87.65, 16: 126.84}
    for R, mean in expect.items():
        got, lo, hi = union_sizes(ref["sel"], R)
        assert abs(got - mean) < 0.01, (R, got)
        assert lo >= 16 and hi <= 16 * R
    # rows per kept block at R = 8: 128 kept (row, block) pairs over ~87.7 distinct blocks
    assert 1.45 < 8 * 16 / union_sizes(ref["sel"], 8)[0] < 1.47


def _bf16(a):
    b = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return (((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(np.float32)


def _worst(n, trials, rng, scale=1 / math.sqrt(128)):
    """Worst max |err| of the attention output with P as one bf16 value and
    with P as bf16 hi + lo, against fp64, over random N(0,1) bf16 inputs with
    n keys."""
    c = scale / math.log(2)
    w1 = w2 = 0.0
    for _ in range(trials):
        q = _bf16(rng.standard_normal(128)).astype(np.float64)
        k = _bf16(rng.standard_normal((n, 128))).astype(np.float64)
        v = _bf16(rng.standard_normal((n, 128))).astype(np.float64)
        s = k @ q
        e = np.exp(scale * (s - s.max()))
        ref = (e / e.sum()) @ v
        x = (s * c).astype(np.float32)
        p = np.exp2(x - x.max()).astype(np.float32)
        hi = _bf16(p)
        lo = _bf16(p - hi)
        l = p.astype(np.float64).sum()
        w1 = max(w1, np.abs((hi.astype(np.float64) @ v) / l - ref).max())
        w2 = max(w2, np.abs(((hi.astype(np.float64) + lo) @ v) / l - ref).max())
    return w1, w2


def test_single_bf16_p_exceeds_the_bound_on_short_rows():
    rng = np.random.default_rng(0)
    one, split = _worst(2, 3000, rng)
    assert one > 2e-3  # a single bf16 P breaks the 2e-3 bound on rows of two keys
    assert split < 1e-5  # the hi + lo split keeps it far inside
    one_long, split_long = _worst(1000, 100, rng)
    assert one_long < 1e-3 and split_long < 1e-5
