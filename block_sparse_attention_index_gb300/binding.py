"""Thin ctypes binding of the C ABI in include/msa.h.

Argument marshalling only: tensors are passed as device pointers, streams as
torch's current CUDA stream, and every step runs in the library's kernels.
There is no CPU fallback: if the compiled library is missing, importing this
module raises.
"""
from __future__ import annotations

import ctypes as C
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmsa_gb300.so")

MSA_OK, MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED, MSA_ERR_WORKSPACE, MSA_ERR_CUDA, MSA_ERR_INTERNAL = range(6)
MSA_OUT_F32, MSA_OUT_BF16 = 0, 1
MSA_KV_BF16, MSA_KV_INT8 = 0, 1
ERR_WAIT_TIMEOUT, ERR_BAD_METADATA, ERR_TMEM_ALLOC = 1, 2, 4

EXPORTED = [
    "msa_status_string", "msa_last_error", "msa_workspace_size", "msa_index_scores", "msa_select_blocks",
    "msa_attend_decode", "msa_attend_prefill", "msa_forward", "msa_forward_marked", "msa_forward_launches",
    "msa_attend_decode_noalloc", "msa_check_wait_timeout",
]


DECODE_MAX_ROWS = 8  # sequences with up to this many rows take the decode kernels


class MsaProblem(C.Structure):
    """Mirror of struct msa_problem."""
    _fields_ = [
        ("num_seqs", C.c_int32), ("num_kv_heads", C.c_int32), ("group_size", C.c_int32),
        ("head_dim", C.c_int32), ("index_dim", C.c_int32), ("block_size", C.c_int32), ("top_k", C.c_int32),
        ("softmax_scale", C.c_float), ("out_dtype", C.c_int32), ("total_rows", C.c_int32),
        ("max_rows_per_seq", C.c_int32), ("max_cache_len", C.c_int32), ("cache_tokens", C.c_int64),
        ("num_decode_seqs", C.c_int32), ("cu_rows", C.c_void_p), ("cache_lens", C.c_void_p),
        ("cache_starts", C.c_void_p), ("block_table", C.c_void_p), ("block_table_stride", C.c_int32),
        ("page_size", C.c_int32), ("index_key_heads", C.c_int32), ("kv_dtype", C.c_int32),
        ("k_scale", C.c_void_p), ("v_scale", C.c_void_p), ("num_decode_rows", C.c_int32),
    ]


class MsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"the MSA CUDA library is not built ({LIB_PATH} is missing); "
                          "run block_sparse_attention_index_gb300.build.build() or __graft_entry__.build()")
    lib = C.CDLL(LIB_PATH)
    P = C.POINTER(MsaProblem)
    vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
    lib.msa_status_string.argtypes = [C.c_int]
    lib.msa_status_string.restype = C.c_char_p
    lib.msa_last_error.argtypes = []
    lib.msa_last_error.restype = C.c_char_p
    lib.msa_workspace_size.argtypes = [P, C.POINTER(C.c_size_t)]
    lib.msa_index_scores.argtypes = [P, vp, vp, vp, i64, vp]
    lib.msa_select_blocks.argtypes = [P, vp, i64, vp, vp, vp]
    lib.msa_attend_decode.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, C.c_size_t, vp]
    lib.msa_attend_prefill.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, C.c_size_t, vp]
    lib.msa_attend_decode_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp]
    lib.msa_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, C.c_size_t, vp]
    lib.msa_forward_marked.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, C.c_size_t, vp,
                                       C.POINTER(vp), i32]
    lib.msa_forward_launches.argtypes = [P]
    lib.msa_check_wait_timeout.argtypes = [vp, C.c_size_t, C.c_uint32, vp]
    lib.msa_forward_launches.restype = i32
    for name in ["msa_workspace_size", "msa_index_scores", "msa_select_blocks", "msa_attend_decode",
                 "msa_attend_decode_noalloc", "msa_check_wait_timeout",
                 "msa_attend_prefill", "msa_forward", "msa_forward_marked"]:
        getattr(lib, name).restype = C.c_int
    return lib


_lib = _load()


def lib():
    return _lib


def _status_name(s: int) -> str:
    return _lib.msa_status_string(s).decode()


def _check(status: int):
    if status != MSA_OK:
        raise MsaError(status, _lib.msa_last_error().decode())


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(device):
    return C.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype, device, shape=None):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


class Problem:
    """A batch description: shapes, host bounds and device metadata.

    seqs_host: list of (n_rows, cache_len); the device metadata (cu_rows,
    cache_lens, cache_starts) is built from it on `device` with the caches
    packed in sequence order unless cache_starts is given.  Paged caches:
    block_table ([B, stride] int32 page numbers, tensor or nested list) and
    page_size, with cache_tokens = rows of the page pool.  ik_heads=1: one
    index key per position shared by every KV head (ik is [T, 1, Di]).
    k_scale, v_scale (float32 [cache_tokens, H] device tensors): the key and
    value caches are int8 with these per-(cache row, head) scales.
    num_decode_rows: host count of decode-family rows ("auto": from seqs_host;
    0: unknown, the decode attention then covers every row slot).
    """

    def __init__(self, H, G, seqs_host, device, top_k=16, scale=None, out_dtype=torch.float32,
                 cache_starts=None, cache_tokens=None, D=128, Di=64, S=64, num_decode_seqs="auto",
                 block_table=None, page_size=0, ik_heads=0, k_scale=None, v_scale=None,
                 num_decode_rows="auto"):
        self.H, self.G, self.D, self.Di, self.S, self.top_k = H, G, D, Di, S, top_k
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.seqs = [(int(n), int(L)) for n, L in seqs_host]
        rows = [n for n, _ in self.seqs]
        lens = [L for _, L in self.seqs]
        cu = [0]
        for n in rows:
            cu.append(cu[-1] + n)
        self.block_table = None
        if block_table is not None:
            if cache_starts is not None or cache_tokens is None:
                raise ValueError("a block table replaces cache_starts and needs cache_tokens (rows of the page pool)")
            self.block_table = torch.as_tensor(block_table, dtype=torch.int32).to(self.device).contiguous()
            if self.block_table.dim() != 2 or self.block_table.shape[0] != len(self.seqs):
                raise ValueError("block_table must be [num_seqs, stride]")
            cache_starts = []
        elif cache_starts is None:
            cache_starts, acc = [], 0
            for L in lens:
                cache_starts.append(acc)
                acc += L
            cache_tokens = acc if cache_tokens is None else cache_tokens
        self.cu_rows = torch.tensor(cu, dtype=torch.int32, device=self.device)
        self.cache_lens = torch.tensor(lens, dtype=torch.int32, device=self.device)
        self.cache_starts = torch.tensor(list(cache_starts), dtype=torch.int64, device=self.device)
        self.total_rows = cu[-1]
        self.cache_tokens = int(cache_tokens)
        self.scale = scale if scale is not None else 1.0 / math.sqrt(D)
        self.out_dtype = out_dtype
        if num_decode_seqs == "auto":
            num_decode_seqs = sum(1 for n in rows if n <= DECODE_MAX_ROWS)
        self.c = MsaProblem(
            len(self.seqs), H, G, D, Di, S, top_k, self.scale,
            MSA_OUT_BF16 if out_dtype == torch.bfloat16 else MSA_OUT_F32,
            self.total_rows, max(rows), max(lens), self.cache_tokens, num_decode_seqs,
            self.cu_rows.data_ptr(), self.cache_lens.data_ptr(),
            self.cache_starts.data_ptr() if self.block_table is None else None,
            None if self.block_table is None else self.block_table.data_ptr(),
            0 if self.block_table is None else int(self.block_table.shape[1]), int(page_size), int(ik_heads))
        if num_decode_rows == "auto":  # rows of the decode-family sequences (1 to 8 rows each)
            num_decode_rows = sum(n for n in rows if n <= DECODE_MAX_ROWS)
        self.c.num_decode_rows = int(num_decode_rows)
        self.KH = 1 if (ik_heads == 1 or H == 1) else H  # index-key heads per position
        if (k_scale is None) != (v_scale is None):
            raise ValueError("k_scale and v_scale go together")
        self.kv_dtype = torch.int8 if k_scale is not None else torch.bfloat16
        self.k_scale = self.v_scale = None
        if k_scale is not None:
            self.k_scale = torch.as_tensor(k_scale, dtype=torch.float32).to(self.device).contiguous()
            self.v_scale = torch.as_tensor(v_scale, dtype=torch.float32).to(self.device).contiguous()
            for t, name in ((self.k_scale, "k_scale"), (self.v_scale, "v_scale")):
                _need(t, name, torch.float32, self.device, (self.cache_tokens, H))
            self.c.kv_dtype = MSA_KV_INT8
            self.c.k_scale = self.k_scale.data_ptr()
            self.c.v_scale = self.v_scale.data_ptr()

    @property
    def max_cache_len(self):
        return self.c.max_cache_len

    def workspace_size(self) -> int:
        n = C.c_size_t(0)
        _check(_lib.msa_workspace_size(C.byref(self.c), C.byref(n)))
        return int(n.value)

    def workspace(self) -> torch.Tensor:
        return torch.empty(self.workspace_size(), dtype=torch.uint8, device=self.device)

    def forward_launches(self) -> int:
        return int(_lib.msa_forward_launches(C.byref(self.c)))

    def new_out(self):
        return torch.empty(self.total_rows, self.H * self.G, self.D, dtype=self.out_dtype, device=self.device)

    def new_sel(self):
        sel = torch.empty(self.total_rows, self.H, self.top_k, dtype=torch.int32, device=self.device)
        nsel = torch.empty(self.total_rows, self.H, dtype=torch.int32, device=self.device)
        return sel, nsel

    # -- checks of the standard layouts
    def _check_q(self, q):
        _need(q, "q", torch.bfloat16, self.device, (self.total_rows, self.H * self.G, self.D))

    def _check_iq(self, iq):
        _need(iq, "iq", torch.bfloat16, self.device, (self.total_rows, self.H, self.Di))

    def _check_cache(self, t, name, width, heads=None):
        dtype = self.kv_dtype if name in ("k", "v") else torch.bfloat16
        _need(t, name, dtype, self.device, (self.cache_tokens, self.H if heads is None else heads, width))

    def _check_sel(self, sel, nsel):
        _need(sel, "sel", torch.int32, self.device, (self.total_rows, self.H, self.top_k))
        _need(nsel, "nsel", torch.int32, self.device, (self.total_rows, self.H))


def index_scores(pb: Problem, iq, ik, ld=None):
    """msa_index_scores: [R, H, ld] fp32 scores (-inf past each row)."""
    pb._check_iq(iq)
    pb._check_cache(ik, "ik", pb.Di, pb.KH)
    ld = ld or ((pb.max_cache_len + 3) // 4 * 4)
    scores = torch.empty(pb.total_rows, pb.H, ld, dtype=torch.float32, device=pb.device)
    _check(_lib.msa_index_scores(C.byref(pb.c), _ptr(iq), _ptr(ik), _ptr(scores), ld, _stream(pb.device)))
    return scores


def select_blocks(pb: Problem, scores):
    """msa_select_blocks: (sel [R,H,top_k], nsel [R,H]) from given scores."""
    _need(scores, "scores", torch.float32, pb.device)
    if scores.dim() != 3 or scores.shape[:2] != (pb.total_rows, pb.H):
        raise ValueError("scores must be [R, H, ld]")
    sel, nsel = pb.new_sel()
    _check(_lib.msa_select_blocks(C.byref(pb.c), _ptr(scores), scores.shape[2], _ptr(sel), _ptr(nsel),
                                  _stream(pb.device)))
    return sel, nsel


def _attend(fn, pb: Problem, q, k, v, sel, nsel, out=None, workspace=None):
    pb._check_q(q)
    pb._check_cache(k, "k", pb.D)
    pb._check_cache(v, "v", pb.D)
    pb._check_sel(sel, nsel)
    out = pb.new_out() if out is None else out
    _need(out, "out", pb.out_dtype, pb.device, (pb.total_rows, pb.H * pb.G, pb.D))
    ws = pb.workspace() if workspace is None else workspace
    _check(fn(C.byref(pb.c), _ptr(q), _ptr(k), _ptr(v), _ptr(sel), _ptr(nsel), _ptr(out), _ptr(ws),
              ws.numel(), _stream(pb.device)))
    return out


def attend_decode(pb: Problem, q, k, v, sel, nsel, out=None, workspace=None):
    """msa_attend_decode: split-KV attention over the given kept blocks."""
    return _attend(_lib.msa_attend_decode, pb, q, k, v, sel, nsel, out, workspace)


def attend_prefill(pb: Problem, q, k, v, sel, nsel, out=None, workspace=None):
    """msa_attend_prefill: tcgen05 attention over the given kept blocks."""
    return _attend(_lib.msa_attend_prefill, pb, q, k, v, sel, nsel, out, workspace)


def attend_decode_noalloc(pb: Problem, q, k, v, sel, nsel, out=None):
    """msa_attend_decode_noalloc: decode attention for callers that cannot
    allocate device memory; the library's fixed scratch replaces the
    workspace (at most 32 sequence x KV-head pairs per call)."""
    pb._check_q(q)
    pb._check_cache(k, "k", pb.D)
    pb._check_cache(v, "v", pb.D)
    pb._check_sel(sel, nsel)
    out = pb.new_out() if out is None else out
    _need(out, "out", pb.out_dtype, pb.device, (pb.total_rows, pb.H * pb.G, pb.D))
    _check(_lib.msa_attend_decode_noalloc(C.byref(pb.c), _ptr(q), _ptr(k), _ptr(v), _ptr(sel), _ptr(nsel),
                                          _ptr(out), _stream(pb.device)))
    return out


def forward(pb: Problem, q, iq, k, v, ik, out=None, sel=None, nsel=None, workspace=None, events=None):
    """msa_forward (msa_forward_marked when events are given).

    Returns (out, sel, nsel); sel/nsel are allocated when not given."""
    pb._check_q(q)
    pb._check_iq(iq)
    pb._check_cache(k, "k", pb.D)
    pb._check_cache(v, "v", pb.D)
    pb._check_cache(ik, "ik", pb.Di, pb.KH)
    out = pb.new_out() if out is None else out
    _need(out, "out", pb.out_dtype, pb.device, (pb.total_rows, pb.H * pb.G, pb.D))
    if sel is None:
        sel, nsel = pb.new_sel()
    pb._check_sel(sel, nsel)
    ws = pb.workspace() if workspace is None else workspace
    args = (C.byref(pb.c), _ptr(q), _ptr(iq), _ptr(k), _ptr(v), _ptr(ik), _ptr(out), _ptr(sel), _ptr(nsel),
            _ptr(ws), ws.numel(), _stream(pb.device))
    if events:
        if any(e is not None and not e.cuda_event for e in events):
            raise ValueError("record each torch.cuda.Event once before passing it (torch creates events lazily)")
        arr = (C.c_void_p * len(events))(*[C.c_void_p(e.cuda_event) if e is not None else None for e in events])
        _check(_lib.msa_forward_marked(*args, arr, len(events)))
    else:
        _check(_lib.msa_forward(*args))
    return out, sel, nsel


def check_wait_timeout(workspace, limit_us: int = 20000):
    """msa_check_wait_timeout: one bounded wait of the library runs out on purpose
    and sets the timeout bit (ERR_WAIT_TIMEOUT) of the workspace's error word."""
    _need(workspace, "workspace", torch.uint8, workspace.device)
    _check(_lib.msa_check_wait_timeout(_ptr(workspace), workspace.numel(), int(limit_us), _stream(workspace.device)))


def error_word(workspace) -> int:
    """The device error word at the start of a workspace (synchronises)."""
    return int(workspace[:4].view(torch.int32).item())


__all__ = ["Problem", "MsaProblem", "MsaError", "index_scores", "select_blocks", "attend_decode", "attend_prefill",
           "attend_decode_noalloc", "check_wait_timeout",
           "forward", "error_word", "lib", "LIB_PATH", "EXPORTED"]
