"""Planted mistakes in the oracle must be caught by its pins.

Each mutant below is a copy of ``oracle/oracle.c`` with one plausible mistake
(a dropped term, a wrong sign, a transposed operand or index, a lost absolute
value, lost precision, a wrong bf16 decode, a row left out between threads).
The copy is compiled on the CPU and the pins of ``_pins.py`` run against it in
a child process; at least one pin has to fail (a crash of the child counts as
caught).  The real oracle is never modified.
"""
import json
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")
TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)

MUTANTS = {
    "wrong_sign": [("accp[j] += a * nrow[j];", "accp[j] -= a * nrow[j];")],
    "dropped_first_term": [("accp[j] += a * nrow[j];", "if (kk > 0) accp[j] += a * nrow[j];")],
    "dropped_last_term": [("accp[j] += a * nrow[j];", "if (kk + 1 < k) accp[j] += a * nrow[j];")],
    "transposed_M_index": [("i * job->ldm + kk", "kk * job->ldm + i")],
    "ignores_ldn": [("oracle_load_row(job->N, job->ntype, kk * job->ldn, n, nrow);",
                     "oracle_load_row(job->N, job->ntype, kk * n, n, nrow);")],
    "D_without_abs": [("accd[j] += abs_a * fabs(nrow[j]);", "accd[j] += a * nrow[j];")],
    "result_rounded_to_fp32": [("job->P[i * job->ldp + j] = accp[j];",
                                "job->P[i * job->ldp + j] = (float)accp[j];")],
    "bf16_wrong_shift": [("<< 16;", "<< 15;")],
    "f32_truncated": [("return (double)((const float *)base)[idx];",
                       "return (double)(long long)((const float *)base)[idx];")],
    "entries_wrong_operand": [("sum += a * b;", "sum += a * a;")],
    "entries_transposed_output": [("const int64_t i = rows[c], j = cols[c];",
                                   "const int64_t i = cols[c], j = rows[c];")],
    "entries_fp32_accumulator": [("double sum = 0.0, sum_abs = 0.0;",
                                  "float sum = 0.0f; double sum_abs = 0.0;")],
    "thread_split_drops_row": [("j->row_end = m * (w + 1) / t;",
                                "j->row_end = m * (w + 1) / t - (w + 1 < t);")],
}

CHILD = r"""
import json, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle, _pins
lib = oracle.load({lib!r})
print(json.dumps(_pins.failing_pins(lib)))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / "oracle_mutant.c"
    path.write_text(src)
    lib = str(tmp_path / "liboracle_mutant.so")
    oracle.compile_library(str(path), lib)
    child = CHILD.format(root=ROOT, tests=TESTS, lib=lib)
    res = subprocess.run([sys.executable, "-c", child], capture_output=True, text=True, timeout=300)
    if res.returncode != 0:
        return  # the mutant crashed the pins: caught
    failed = json.loads(res.stdout.strip().splitlines()[-1])
    assert failed, f"mutant {name} passed every pin"
