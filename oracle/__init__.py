"""CPU oracle for the MSA hot path (fp64, plain C) -- TEST INFRASTRUCTURE.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may
import this package.  It shares no code with the CUDA path and never imports
it; the two meet only in the seeded inputs drawn by ``synth``.

Every function follows the definition in ``msa_oracle.c`` (index scores,
max-pool, top-k with the forced local block, softmax attention over the kept
blocks), each step citing the passage of the pages it restates.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_libs = {}


class _Problem(C.Structure):
    _fields_ = [
        ("num_seqs", C.c_int32), ("H", C.c_int32), ("G", C.c_int32), ("D", C.c_int32),
        ("Di", C.c_int32), ("S", C.c_int32), ("top_k", C.c_int32), ("scale", C.c_double),
        ("cu_rows", C.c_void_p), ("cache_lens", C.c_void_p), ("cache_starts", C.c_void_p),
        ("ik_heads", C.c_int32), ("kv_int8", C.c_int32), ("k_scale", C.c_void_p), ("v_scale", C.c_void_p),
    ]


def lib(path: str | None = None):
    """The oracle library (the default build, or another build at `path`)."""
    key = path or ""
    if key not in _libs:
        L = C.CDLL(path or _build.build())
        P = C.POINTER(_Problem)
        vp, i64, i32 = C.c_void_p, C.c_int64, C.c_int32
        L.oracle_index_scores.argtypes = [P, vp, vp, i64, i32, vp, i64]
        L.oracle_index_scores.restype = C.c_int
        L.oracle_pool.argtypes = [vp, i64, i32, vp]
        L.oracle_pool.restype = C.c_int
        L.oracle_select.argtypes = [vp, i32, i32, vp]
        L.oracle_select.restype = C.c_int
        L.oracle_attend.argtypes = [P, vp, vp, vp, i64, i32, vp, i32, vp]
        L.oracle_attend.restype = C.c_int
        L.oracle_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp, i64, i32]
        L.oracle_forward.restype = C.c_int
        L.oracle_num_threads.restype = C.c_int
        _libs[key] = L
    return _libs[key]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


class Problem:
    """Shape and metadata of one MSA problem (arrays are kept alive here)."""

    def __init__(self, H, G, cu_rows, cache_lens, cache_starts, D=128, Di=64, S=64, top_k=16, scale=None,
                 ik_heads=None, k_scale=None, v_scale=None):
        self.cu_rows = np.ascontiguousarray(cu_rows, dtype=np.int32)
        self.cache_lens = np.ascontiguousarray(cache_lens, dtype=np.int32)
        self.cache_starts = np.ascontiguousarray(cache_starts, dtype=np.int64)
        self.H, self.G, self.D, self.Di, self.S, self.top_k = H, G, D, Di, S, top_k
        self.scale = scale if scale is not None else 1.0 / np.sqrt(D)
        self.ik_heads = H if ik_heads is None else ik_heads  # 1: one index key shared by all KV heads
        # int8 key/value cache: one float scale per (cache row, KV head) for each of k and v
        self.kv_int8 = k_scale is not None
        if self.kv_int8 != (v_scale is not None):
            raise ValueError("k_scale and v_scale go together")
        self.k_scale = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
        self.v_scale = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float32)
        self.c = _Problem(len(self.cache_lens), H, G, D, Di, S, top_k, self.scale,
                          _ptr(self.cu_rows), _ptr(self.cache_lens), _ptr(self.cache_starts), self.ik_heads,
                          int(self.kv_int8), _ptr(self.k_scale), _ptr(self.v_scale))

    @classmethod
    def from_workload(cls, w, x):
        return cls(w.H, w.G, x["cu_rows"], x["cache_lens"], x["cache_starts"], D=w.D, Di=w.Di,
                   S=w.S, top_k=w.top_k, scale=w.softmax_scale, ik_heads=int(x["ik"].shape[1]),
                   k_scale=x.get("k_scale"), v_scale=x.get("v_scale"))

    @property
    def total_rows(self):
        return int(self.cu_rows[-1])

    def position(self, r):
        b = int(np.searchsorted(self.cu_rows, r, side="right") - 1)
        n = int(self.cu_rows[b + 1] - self.cu_rows[b])
        return b, int(self.cache_lens[b]) - n + (r - int(self.cu_rows[b]))

    def max_blocks(self):
        return int((int(self.cache_lens.max()) + self.S - 1) // self.S)


def _u16(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint16)


def _kv(pr: Problem, a):
    """A key or value cache as the oracle reads it: int8 values when the
    problem has scales, bf16 bit patterns otherwise."""
    if a is None:
        return None
    if pr.kv_int8:
        if a.dtype != np.int8:
            raise ValueError("an int8 key/value cache needs int8 values")
        return np.ascontiguousarray(a)
    return _u16(a)


def index_scores(pr: Problem, iq, ik, r: int, h: int, lib_path=None) -> np.ndarray:
    """s_t for t = 0..p of row r and KV head h (fp64)."""
    _, p = pr.position(r)
    s = np.empty(p + 1, dtype=np.float64)
    iq, ik = _u16(iq), _u16(ik)
    n = lib(lib_path).oracle_index_scores(C.byref(pr.c), _ptr(iq), _ptr(ik), r, h, _ptr(s), len(s))
    assert n == p + 1, "oracle disagrees on the row's position"
    return s


def pool(s, S: int = 64, lib_path=None) -> np.ndarray:
    """Block max-pool of a score vector over blocks of S positions."""
    s = np.ascontiguousarray(s, dtype=np.float64)
    m = np.empty((len(s) + S - 1) // S, dtype=np.float64)
    n = lib(lib_path).oracle_pool(_ptr(s), len(s), S, _ptr(m))
    assert n == len(m)
    return m


def select(m, top_k: int = 16, lib_path=None):
    """Kept blocks (ascending) from pooled scores; the last block is the forced
    local block.  Returns (sel padded with -1 to top_k, nsel)."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    sel = np.empty(top_k, dtype=np.int32)
    n = lib(lib_path).oracle_select(_ptr(m), len(m), top_k, _ptr(sel))
    return sel, n


def attend(pr: Problem, q, k, v, r: int, h: int, sel, lib_path=None) -> np.ndarray:
    """[G, D] fp64 output of the G query heads of KV head h at row r over the
    listed blocks (entries < 0 ignored)."""
    sel = np.ascontiguousarray([s for s in np.asarray(sel).ravel() if s >= 0], dtype=np.int32)
    out = np.empty((pr.G, pr.D), dtype=np.float64)
    q, k, v = _u16(q), _kv(pr, k), _kv(pr, v)
    nk = lib(lib_path).oracle_attend(C.byref(pr.c), _ptr(q), _ptr(k), _ptr(v), r, h, _ptr(sel), len(sel), _ptr(out))
    assert nk >= 0
    return out


def forward(pr: Problem, x: dict, rows=None, threads: int = 0, with_out: bool = True, with_pooled: bool = False, lib_path=None):
    """Steps 1-4 for the listed rows (all when rows is None).

    Returns dict(sel [n,H,top_k] int32, nsel [n,H] int32, out [n,H*G,D] fp64 or
    None, pooled [n,H,max_blocks] fp64 or None, rows)."""
    R = pr.total_rows
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = R if rows_arr is None else len(rows_arr)
    H = pr.H
    sel = np.empty((n, H, pr.top_k), dtype=np.int32)
    nsel = np.empty((n, H), dtype=np.int32)
    out = np.empty((n, H * pr.G, pr.D), dtype=np.float64) if with_out else None
    mb = pr.max_blocks()
    pooled = np.empty((n, H, mb), dtype=np.float64) if with_pooled else None
    q, iq, ik = _u16(x["q"]), _u16(x["iq"]), _u16(x["ik"])
    k, v = _kv(pr, x.get("k")), _kv(pr, x.get("v"))
    if with_out and (k is None or v is None):
        raise ValueError("k and v are needed for the attention output")
    rc = lib(lib_path).oracle_forward(C.byref(pr.c), _ptr(q), _ptr(iq), _ptr(k), _ptr(v), _ptr(ik), _ptr(rows_arr), n,
                              _ptr(sel), _ptr(nsel), _ptr(out), _ptr(pooled), mb, threads)
    if rc != 0:
        raise ValueError("oracle: a listed row does not belong to any sequence")
    return dict(sel=sel, nsel=nsel, out=out, pooled=pooled,
                rows=np.arange(R) if rows_arr is None else rows_arr)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


__all__ = ["Problem", "index_scores", "pool", "select", "attend", "forward", "num_threads", "lib"]
