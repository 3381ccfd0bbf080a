"""Planted controls: oracle builds with one deliberate mistake each must fail
at least one pin (after the kernel-contract idea of planted controls that
must go red, minimax_m3 CUDA backend PR #1388, "How it was checked").

The mistakes are planted in a temporary copy of the oracle source, on the
CPU; the oracle itself is never modified."""
import os
import shutil
import subprocess

import pytest

import helpers

SRC = os.path.join(helpers.ROOT, "oracle", "msa_oracle.c")

MUTANTS = {
    "drop_forced_local": [("    sel[n++] = J;\n", ""),
                          ("int32_t others = top_k - 1 < J ? top_k - 1 : J;", "int32_t others = top_k < J ? top_k : J;")],
    "flip_tie_break": [("return (x->j < y->j) ? -1 : (x->j > y->j);", "return (x->j > y->j) ? -1 : (x->j < y->j);")],
    "no_causal_rows": [("*p_out = (int64_t)pr->cache_lens[b] - n + i;", "*p_out = (int64_t)pr->cache_lens[b] - 1 + 0 * (n + i);")],
    "unscaled_logits": [("x[i] = pr->scale * acc;", "x[i] = acc;")],
    "wrong_index_key_head": [("* kh + (kh == 1 ? 0 : h))", "* kh + 0)")],
    "unnormalised_output": [("o[d] = nk > 0 ? o[d] / den : 0.0;", "o[d] = nk > 0 ? o[d] : 0.0;")],
    "last_not_max_pool": [("if (s[t] > best) best = s[t];", "best = s[t];")],
    "values_from_keys": [("kv_value(pr, v, pr->v_scale", "kv_value(pr, k, pr->v_scale")],
    "int8_scale_ignored": [("return (double)scale[row * pr->H + h] * (double)((const int8_t*)base)[i];",
                            "return (double)((const int8_t*)base)[i];")],
    "int8_key_scale_for_values": [("kv_value(pr, v, pr->v_scale", "kv_value(pr, v, pr->k_scale")],
    "int8_scale_of_head_0": [("scale[row * pr->H + h]", "scale[row * pr->H]")],
    "block_end_off_by_one": [("t < (int64_t)(sel[i] + 1) * S;", "t < (int64_t)(sel[i] + 1) * S - 1;")],
    "drops_current_position": [("if (t >= 0 && t <= p) keys[nk++] = t;", "if (t >= 0 && t < p) keys[nk++] = t;")],
    "min_not_max_selection": [("if (x->m > y->m) return -1;\n    if (x->m < y->m) return 1;",
                               "if (x->m < y->m) return -1;\n    if (x->m > y->m) return 1;")],
}


def _build(tmp_path, name, patches):
    src = open(SRC).read()
    for old, new in patches:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-shared", "-fPIC", str(c), "-o", str(so), "-lm"], check=True,
                   capture_output=True)
    return str(so)


def _failing_checks(lib_path):
    failed = []
    for check in helpers.ALL_CHECKS:
        try:
            check(lib_path=lib_path)
        except AssertionError:
            failed.append(check.__name__)
    return failed


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_unmutated_copy_passes(tmp_path):
    assert _failing_checks(_build(tmp_path, "clean", [])) == []


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    failed = _failing_checks(_build(tmp_path, name, MUTANTS[name]))
    assert failed, f"planted mistake {name} passed every pin"
