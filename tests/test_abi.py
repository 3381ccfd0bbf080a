"""The C ABI without a GPU: the library loads, exports every function that
include/msa.h declares, the ctypes struct mirrors the C struct byte for byte,
and invalid arguments are rejected on the host before anything is enqueued."""
import ctypes as C
import os
import re
import shutil
import subprocess

import pytest

import helpers

HEADER = os.path.join(helpers.ROOT, "include", "msa.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    import block_sparse_attention_index_gb300 as m
    declared = _declared_functions()
    assert set(declared) == set(m.EXPORTED), (declared, m.EXPORTED)
    for name in declared:
        assert hasattr(m.lib(), name), name


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_struct_layout_matches_header(tmp_path):
    import block_sparse_attention_index_gb300 as m
    fields = [f for f, _ in m.MsaProblem._fields_]
    prog = "#include <stdio.h>\n#include <stddef.h>\n#include \"msa.h\"\nint main(void){\n"
    prog += 'printf("%zu\\n", sizeof(msa_problem));\n'
    for f in fields:
        prog += f'printf("%zu\\n", offsetof(msa_problem, {f}));\n'
    prog += "return 0;}\n"
    (tmp_path / "t.c").write_text(prog)
    exe = tmp_path / "t"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(tmp_path / "t.c"), "-o", str(exe)], check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert vals[0] == C.sizeof(m.MsaProblem)
    assert vals[1:] == [getattr(m.MsaProblem, f).offset for f in fields]


def _problem(**over):
    import block_sparse_attention_index_gb300 as m
    vals = dict(num_seqs=1, num_kv_heads=4, group_size=16, head_dim=128, index_dim=64, block_size=64, top_k=16,
                softmax_scale=0.088, out_dtype=0, total_rows=1, max_rows_per_seq=1, max_cache_len=4096,
                cache_tokens=4096, num_decode_seqs=1, cu_rows=256, cache_lens=512, cache_starts=768)
    vals.update(over)
    return m.MsaProblem(**vals)


@pytest.mark.parametrize("over,status", [
    (dict(head_dim=64), 2), (dict(index_dim=32), 2), (dict(block_size=128), 2), (dict(top_k=17), 2),
    (dict(top_k=0), 1), (dict(group_size=17), 2), (dict(group_size=0), 1), (dict(num_kv_heads=3), 2),
    (dict(num_seqs=0), 1), (dict(softmax_scale=float("nan")), 1), (dict(softmax_scale=-1.0), 1),
    (dict(out_dtype=7), 1), (dict(total_rows=0), 1), (dict(max_rows_per_seq=2), 1),
    (dict(max_cache_len=(1 << 21) + 1), 2), (dict(cache_tokens=0), 1), (dict(num_decode_seqs=2), 1),
    (dict(cu_rows=None), 1), (dict(cu_rows=258), 1), (dict(cache_lens=258), 1), (dict(cache_starts=260), 1),
    (dict(cache_starts=None), 1),
    (dict(num_seqs=2, max_rows_per_seq=8, total_rows=9, num_decode_seqs=1), 1),  # <= 8 rows: all decode family
    # paged caches: page size a power of two >= 64, pool a whole number of pages,
    # table wide enough for max_cache_len, table aligned
    (dict(cache_starts=None, block_table=1024, block_table_stride=64, page_size=32), 2),
    (dict(cache_starts=None, block_table=1024, block_table_stride=64, page_size=96), 2),
    (dict(cache_starts=None, block_table=1024, block_table_stride=64, page_size=64, cache_tokens=4000), 1),
    (dict(cache_starts=None, block_table=1024, block_table_stride=63, page_size=64), 1),
    (dict(cache_starts=None, block_table=1026, block_table_stride=64, page_size=64), 1),
    # int8 key/value cache: a known element type, both scale arrays, 4-byte aligned
    (dict(kv_dtype=2), 1), (dict(kv_dtype=1), 1), (dict(kv_dtype=1, k_scale=2048), 1),
    (dict(kv_dtype=1, k_scale=2048, v_scale=2050), 1),
    # host count of decode-family rows: within the rows and 1..8 per decode sequence
    (dict(num_decode_rows=2), 1), (dict(num_seqs=2, total_rows=20, max_rows_per_seq=16, num_decode_seqs=1,
                                        num_decode_rows=9), 1),
])
def test_invalid_problem_rejected_on_host(over, status):
    import block_sparse_attention_index_gb300 as m
    n = C.c_size_t(0)
    pb = _problem(**over)
    assert m.lib().msa_workspace_size(C.byref(pb), C.byref(n)) == status
    assert m.lib().msa_last_error()


def test_int8_problem_accepted_on_host():
    import block_sparse_attention_index_gb300 as m
    n = C.c_size_t(0)
    pb = _problem(kv_dtype=1, k_scale=2048, v_scale=4096)
    assert m.lib().msa_workspace_size(C.byref(pb), C.byref(n)) == 0, m.lib().msa_last_error()


def test_workspace_size_and_pointer_checks():
    import block_sparse_attention_index_gb300 as m
    L = m.lib()
    pb = _problem()
    n = C.c_size_t(0)
    assert L.msa_workspace_size(C.byref(pb), C.byref(n)) == 0
    assert n.value > 0 and n.value % 256 == 0
    ws = C.c_void_p(1 << 20)
    fake = C.c_void_p(1 << 30)
    # null q, misaligned out, undersized and misaligned workspace: all rejected before any CUDA call
    assert L.msa_forward(C.byref(pb), None, fake, fake, fake, fake, fake, None, None, ws, n.value, None) == 1
    assert L.msa_forward(C.byref(pb), fake, fake, fake, fake, fake, C.c_void_p((1 << 30) + 4), None, None, ws,
                         n.value, None) == 1
    assert L.msa_forward(C.byref(pb), fake, fake, fake, fake, fake, fake, None, None, ws, n.value - 256, None) == 3
    assert L.msa_forward(C.byref(pb), fake, fake, fake, fake, fake, fake, None, None, C.c_void_p((1 << 20) + 16),
                         n.value, None) == 3
    assert L.msa_forward(C.byref(pb), fake, fake, fake, fake, fake, fake, fake, None, ws, n.value, None) == 1
    pb2 = _problem(max_rows_per_seq=1, total_rows=2, num_seqs=2, num_decode_seqs=2)
    assert L.msa_attend_decode(C.byref(pb2), fake, fake, fake, None, fake, fake, ws, 1 << 30, None) == 1
    assert L.msa_index_scores(C.byref(pb), fake, fake, fake, 100, None) == 1  # ld < max_cache_len
    # the wait check: null workspace, no room for the error word, a limit outside [1 us, 2 s]
    assert L.msa_check_wait_timeout(None, 256, 1000, None) == 1
    assert L.msa_check_wait_timeout(ws, 2, 1000, None) == 3
    assert L.msa_check_wait_timeout(ws, 256, 0, None) == 1
    assert L.msa_check_wait_timeout(ws, 256, 2000001, None) == 1
    assert L.msa_forward_launches(C.byref(pb)) == 2
    assert L.msa_forward_launches(C.byref(_problem(max_rows_per_seq=12, total_rows=12, num_decode_seqs=0))) == 2
    assert L.msa_forward_launches(C.byref(_problem(num_seqs=2, max_rows_per_seq=9, total_rows=10,
                                                   num_decode_seqs=1))) == 4
    # up to 8 rows per sequence is the decode family alone
    assert L.msa_forward_launches(C.byref(_problem(num_seqs=2, max_rows_per_seq=8, total_rows=9,
                                                   num_decode_seqs=2))) == 2


def test_paged_problem_accepted_on_host():
    import block_sparse_attention_index_gb300 as m
    n = C.c_size_t(0)
    for ps, stride in ((64, 64), (256, 16), (4096, 1)):
        pb = _problem(cache_starts=None, block_table=1024, block_table_stride=stride, page_size=ps)
        assert m.lib().msa_workspace_size(C.byref(pb), C.byref(n)) == 0, m.lib().msa_last_error()
