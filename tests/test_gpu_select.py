"""Block selection from crafted pooled scores (msa_select_blocks), against the
oracle's selection on the same scores: bit-exact.  The patterns drive every
branch of the CTA selection: a handful of candidates above the bound,
hundreds of them (threads whose every score beats the others' best), more
than the candidate list holds (the arg-max rounds), all-equal and
few-valued scores (ties everywhere), and rows longer than the scores kept in
registers.  Scores are constant over each 64-position block, so the pooled
score of block j is the crafted value."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import msa

pytestmark = pytest.mark.gpu

NT = 128  # threads of the selecting CTA; lane l of warp w holds blocks j = 32w + l + 128 i


def crafted(kind, J, rng):
    m = rng.standard_normal(J).astype(np.float32) * 100.0  # j < J; block J is the local one
    j = np.arange(J)
    lane0 = j % NT  # thread holding block j
    if kind == "wide":  # threads 0..13 hold only high scores, thread 14's best sits just under them
        hi = lane0 < 14
        m[hi] = 3000.0 + j[hi]
        m[lane0 == 14] = 2999.0
    elif kind == "equal":
        m[:] = 7.0
    elif kind == "integer":  # few distinct values: many ties at the bound
        m = rng.integers(-3, 4, J).astype(np.float32)
    elif kind == "descending":
        m = (J - j).astype(np.float32)
    return m


@pytest.mark.parametrize("kind", ["random", "wide", "equal", "integer", "descending"])
@pytest.mark.parametrize("J", [16, 40, 1023, 4000, 5000])
def test_select_crafted(kind, J):
    m_ = msa()
    rng = np.random.default_rng(J * 7 + len(kind))
    L = J * 64 + 1 + int(rng.integers(0, 63))  # the local block J holds the row's position
    pooled = crafted(kind, J, rng)
    pb = m_.Problem(1, 16, [(1, L)], "cuda")
    ld = (L + 3) // 4 * 4
    s = np.full(ld, -np.inf, dtype=np.float32)
    s[:J * 64] = np.repeat(pooled, 64)
    s[J * 64:L] = rng.standard_normal(L - J * 64).astype(np.float32)
    sel, nsel = m_.select_blocks(pb, torch.from_numpy(s).view(1, 1, ld).cuda())
    torch.cuda.synchronize()
    ref_sel, ref_n = oracle.select(oracle.pool(s[:L].astype(np.float64)), 16)
    assert int(nsel[0, 0]) == ref_n
    assert sel[0, 0].cpu().numpy().tolist() == ref_sel.tolist()
