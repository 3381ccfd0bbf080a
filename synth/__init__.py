"""Seeded synthetic inputs for the MSA hot path.

This module is shared by the CPU oracle (``oracle/``), the tests and the
benchmark.  It holds no step of the method's arithmetic: it only draws the
bytes that both sides consume (bf16 q/k/v, integer-valued bf16 index q/k)
and the per-sequence metadata (rows per sequence, cache lengths, where each
sequence's cache starts).

Generator: counter-based splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014): value i of stream s under
seed x is mix64(key(x, s) + (i + 1) * 0x9E3779B97F4A7C15).  Uniform doubles
take the top 53 bits.  Normals use the Box-Muller transform on consecutive
pairs of uniforms and are rounded double -> float -> bf16, each step
round-to-nearest-even.  Index q/k are uniform integers in [-8, 8], stored
as bf16 (exact), so fp32 index scores are exact.  An int8 key/value cache
(kv_dtype "int8") holds uniform integers in [-127, 127] with one float32
scale per (cache row, KV head) drawn uniformly from [0.5/64, 1.5/64], so the
dequantised values have about the spread of the bf16 N(0,1) cache.

Layouts (all row-major, bf16 carried as uint16 bit patterns):
  q   [total_rows, H*G, D]     query row r, q head h*G+g
  iq  [total_rows, H, Di]      index query
  k,v [cache_tokens, H, D]     sequence b occupies rows cache_starts[b] .. +L_b
  ik  [cache_tokens, H, Di]    index keys, same token rows as k/v
  k_scale, v_scale [cache_tokens, H] float32 (int8 caches only)
Row i of a sequence with n rows and cache length L sits at position L-n+i.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "make_inputs", "WORKLOADS", "workload", "bf16_to_f32",
    "uniform", "normal_bf16", "int_bf16", "int8_values", "uniform_f32", "ragged_lengths",
]

_MASK = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_CHUNK = 1 << 20

# stream ids, one per drawn tensor
STREAM_Q, STREAM_IQ, STREAM_K, STREAM_V, STREAM_IK, STREAM_LENS = 1, 2, 3, 4, 5, 6
STREAM_KSCALE, STREAM_VSCALE = 7, 8


def _mix_int(z: int) -> int:
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def _key(seed: int, stream: int) -> int:
    return _mix_int(seed * _GOLDEN + stream * 0xD1B54A32D192ED03 + 1)


def _bits(key: int, start: int, n: int) -> np.ndarray:
    """splitmix64 outputs for counters start .. start+n-1 (uint64)."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    z = i * np.uint64(_GOLDEN) + np.uint64(key)
    z ^= z >> np.uint64(30)
    z *= np.uint64(_M1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(_M2)
    z ^= z >> np.uint64(31)
    return z


def _u53(bits: np.ndarray) -> np.ndarray:
    return (bits >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n uniform doubles in [0, 1)."""
    return _u53(_bits(_key(seed, stream), start, n))


def _f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    f = x.astype(np.float32).view(np.uint32)
    r = (f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _parallel(fn, total: int, step: int) -> None:
    starts = range(0, total, step)
    if total <= step:
        for s in starts:
            fn(s)
        return
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(fn, starts))


def normal_bf16(seed: int, stream: int, shape) -> np.ndarray:
    """N(0,1) draws rounded to bf16, returned as uint16 bit patterns."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint16)
    key = _key(seed, stream)
    npairs = (n + 1) // 2

    def one(p0):
        m = min(_CHUNK, npairs - p0)
        u = _u53(_bits(key, 2 * p0, 2 * m)).reshape(m, 2)
        rad = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
        ang = (2.0 * math.pi) * u[:, 1]
        z = np.empty((m, 2), dtype=np.float64)
        z[:, 0] = rad * np.cos(ang)
        z[:, 1] = rad * np.sin(ang)
        zf = z.reshape(-1)
        lo, hi = 2 * p0, min(n, 2 * (p0 + m))
        out[lo:hi] = _f64_to_bf16_bits(zf[: hi - lo])

    _parallel(one, npairs, _CHUNK)
    return out.reshape(shape)


def int_bf16(seed: int, stream: int, shape, lo: int = -8, hi: int = 8) -> np.ndarray:
    """Uniform integers in [lo, hi] stored as bf16 bit patterns."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint16)
    key = _key(seed, stream)
    span = hi - lo + 1

    def one(s0):
        m = min(_CHUNK, n - s0)
        u = _u53(_bits(key, s0, m))
        v = np.floor(u * span) + lo
        out[s0:s0 + m] = _f64_to_bf16_bits(v)

    _parallel(one, n, _CHUNK)
    return out.reshape(shape)


def int8_values(seed: int, stream: int, shape, lo: int = -127, hi: int = 127) -> np.ndarray:
    """Uniform integers in [lo, hi] as int8."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.int8)
    key = _key(seed, stream)
    span = hi - lo + 1

    def one(s0):
        m = min(_CHUNK, n - s0)
        u = _u53(_bits(key, s0, m))
        out[s0:s0 + m] = (np.floor(u * span) + lo).astype(np.int8)

    _parallel(one, n, _CHUNK)
    return out.reshape(shape)


def uniform_f32(seed: int, stream: int, shape, lo: float, hi: float) -> np.ndarray:
    """Uniform draws in [lo, hi) rounded to float32."""
    n = int(np.prod(shape, dtype=np.int64))
    u = uniform(seed, stream, n)
    return (lo + (hi - lo) * u).astype(np.float32).reshape(shape)


def ragged_lengths(seed: int, n: int, lo: int, hi: int) -> list[int]:
    """n lengths drawn log-uniformly from [lo, hi)."""
    u = uniform(seed, STREAM_LENS, n)
    a, b = math.log(lo), math.log(hi)
    return [int(math.floor(math.exp(a + x * (b - a)))) for x in u]


@dataclass
class Workload:
    """One seeded synthetic MSA problem.

    seqs: list of (n_rows, L): n query rows at positions L-n .. L-1 against a
    cache of L tokens (the rows' own tokens included).
    """
    name: str
    H: int
    G: int
    seqs: list
    D: int = 128
    Di: int = 64
    S: int = 64
    top_k: int = 16
    seed: int = 0
    scale: float | None = None
    note: str = ""
    extra: dict = field(default_factory=dict)
    ik_heads: int = 0  # index keys per position: 0 = one per KV head, 1 = one shared by all heads
    kv_dtype: str = "bf16"  # "int8": int8 key/value cache with a float32 scale per (cache row, KV head)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def total_rows(self) -> int:
        return sum(n for n, _ in self.seqs)

    @property
    def cache_tokens(self) -> int:
        return sum(L for _, L in self.seqs)

    @property
    def num_seqs(self) -> int:
        return len(self.seqs)


def make_inputs(w: Workload, with_kv: bool = True) -> dict:
    """Draw every input of workload w.  Returns numpy arrays (bf16 as uint16)."""
    B = w.num_seqs
    rows = np.array([n for n, _ in w.seqs], dtype=np.int64)
    lens = np.array([L for _, L in w.seqs], dtype=np.int64)
    if np.any(rows < 1) or np.any(rows > lens):
        raise ValueError("each sequence needs 1 <= n_rows <= L")
    cu_rows = np.zeros(B + 1, dtype=np.int32)
    cu_rows[1:] = np.cumsum(rows)
    starts = np.zeros(B, dtype=np.int64)
    starts[1:] = np.cumsum(lens)[:-1]
    R, T = int(cu_rows[-1]), int(lens.sum())
    out = dict(
        cu_rows=cu_rows,
        cache_lens=lens.astype(np.int32),
        cache_starts=starts,
        q=normal_bf16(w.seed, STREAM_Q, (R, w.H * w.G, w.D)),
        iq=int_bf16(w.seed, STREAM_IQ, (R, w.H, w.Di)),
        ik=int_bf16(w.seed, STREAM_IK, (T, 1 if w.ik_heads == 1 else w.H, w.Di)),
    )
    if with_kv and w.kv_dtype == "int8":
        out["k"] = int8_values(w.seed, STREAM_K, (T, w.H, w.D))
        out["v"] = int8_values(w.seed, STREAM_V, (T, w.H, w.D))
        out["k_scale"] = uniform_f32(w.seed, STREAM_KSCALE, (T, w.H), 0.5 / 64, 1.5 / 64)
        out["v_scale"] = uniform_f32(w.seed, STREAM_VSCALE, (T, w.H), 0.5 / 64, 1.5 / 64)
    elif with_kv:
        out["k"] = normal_bf16(w.seed, STREAM_K, (T, w.H, w.D))
        out["v"] = normal_bf16(w.seed, STREAM_V, (T, w.H, w.D))
    return out


STREAM_PAGES, STREAM_POOL = 101, 102


def paged_layout(w: Workload, x: dict, page_size: int, spare_pages: int = 3, seed: int = 0) -> dict:
    """The same caches as a page pool: sequence b's positions [i*page, (i+1)*page)
    live on page table[b, i] of the pool, the pages shuffled by a seeded
    permutation; pool rows that hold no position (page tails, spare pages) get
    other random values, so that reading a wrong row changes the result.
    Returns pool arrays k, v, ik ([num_pages * page_size, H, width]), the block
    table [B, stride] int32 (-1 past each sequence) and num_pages."""
    lens = [int(L) for _, L in w.seqs]
    pages = [(L + page_size - 1) // page_size for L in lens]
    num_pages = sum(pages) + spare_pages
    stride = max(pages)
    order = np.argsort(uniform(seed, STREAM_PAGES, num_pages))  # a seeded permutation of the pages
    table = np.full((len(lens), stride), -1, dtype=np.int32)
    nxt = 0
    for b, npg in enumerate(pages):
        table[b, :npg] = order[nxt:nxt + npg]
        nxt += npg
    rows = num_pages * page_size
    out = dict(table=table, num_pages=num_pages, page_size=page_size)
    starts = x["cache_starts"]
    for i, name in enumerate(n for n in ("k", "v", "ik", "k_scale", "v_scale") if n in x):
        src = x[name]
        if name == "ik":
            pool = int_bf16(seed, STREAM_POOL + i, (rows,) + src.shape[1:])
        elif src.dtype == np.int8:
            pool = int8_values(seed, STREAM_POOL + i, (rows,) + src.shape[1:])
        elif src.dtype == np.float32:
            pool = uniform_f32(seed, STREAM_POOL + i, (rows,) + src.shape[1:], 0.5 / 64, 1.5 / 64)
        else:
            pool = normal_bf16(seed, STREAM_POOL + i, (rows,) + src.shape[1:])
        for b, L in enumerate(lens):
            for pg in range(pages[b]):
                t0, t1 = pg * page_size, min(L, (pg + 1) * page_size)
                r0 = int(table[b, pg]) * page_size
                pool[r0:r0 + (t1 - t0)] = src[int(starts[b]) + t0:int(starts[b]) + t1]
        out[name] = pool
    return out


def _c5_seqs(seed: int) -> list:
    lens = ragged_lengths(seed, 8, 1024, 196608)
    return [(1, L) for L in lens] + [(512, 32768 + 512)]


# The five measured workloads: head layout 4 KV x 16 query heads (1 x 16 for the
# first), head_dim 128, index dim 64, block 64, top-16 with the local block forced.
WORKLOADS = {
    "decode_1x4096": lambda: Workload("decode_1x4096", H=1, G=16, seqs=[(1, 4096)],
                                      note="decode, 1 row, 1 KV head x 16 q heads, 4,096 cached tokens"),
    "decode_4x65536": lambda: Workload("decode_4x65536", H=4, G=16, seqs=[(1, 65536)] * 4,
                                       note="decode batch 4, 65,536 cached tokens each, 4 KV x 16 q heads"),
    "prefill_4096_at_8192": lambda: Workload("prefill_4096_at_8192", H=4, G=16, seqs=[(4096, 8192 + 4096)],
                                             note="prefill chunk of 4,096 rows after an 8,192-token prefix"),
    "decode_1x262144": lambda: Workload("decode_1x262144", H=4, G=16, seqs=[(1, 262144)],
                                        note="long-context decode, 262,144 cached tokens"),
    "mixed_8dec_512pre": lambda: Workload("mixed_8dec_512pre", H=4, G=16, seqs=_c5_seqs(0),
                                          note="8 ragged decode rows (log-uniform 1,024..196,608) + a 512-row chunk at 32,768"),
    # beyond the five configurations: drafted windows (several decode rows per sequence)
    "decode_4x4_65536": lambda: Workload("decode_4x4_65536", H=4, G=16, seqs=[(4, 65536)] * 4,
                                         note="drafted windows: 4 sequences x 4 rows, 65,536 cached tokens each"),
    "decode_4x65536_shared_ik": lambda: Workload("decode_4x65536_shared_ik", H=4, G=16, seqs=[(1, 65536)] * 4,
                                                 ik_heads=1,
                                                 note="decode batch 4 at 65,536, one index key per position shared by the 4 KV heads"),
    "decode_4x65536_int8": lambda: Workload("decode_4x65536_int8", H=4, G=16, seqs=[(1, 65536)] * 4,
                                            kv_dtype="int8",
                                            note="decode batch 4 at 65,536 with an int8 key/value cache "
                                                 "(a float32 scale per position and KV head)"),
    "prefill_4096_at_8192_int8": lambda: Workload("prefill_4096_at_8192_int8", H=4, G=16,
                                                  seqs=[(4096, 8192 + 4096)], kv_dtype="int8",
                                                  note="prefill chunk of 4,096 rows after an 8,192-token prefix, "
                                                       "int8 key/value cache"),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]()
