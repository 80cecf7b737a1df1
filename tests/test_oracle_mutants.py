"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one.

Each mutant is a one-line textual change of ``oracle/pkv_oracle.c`` (a
dropped term, a wrong sign, index or operand), compiled to a temporary
library and loaded by a fresh pytest process through ``PKV_ORACLE_SO``.  The
pin suite must fail for each of them; the unmutated source must pass.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, original text, replacement, which occurrence: 0-based or None for all)
MUTANTS = [
    ("gqa_mapping_decode", "h / group", "h % n_kv_heads", 0),
    ("gqa_mapping_prefill", "h / group", "h % n_kv_heads", 1),
    ("scale_dropped", "scores[j] = scale * dot;", "scores[j] = dot;", None),
    ("softmax_sign", "exp(scores[j] - m)", "exp(m - scores[j])", None),
    ("causal_off_by_one", "(kv_len - q_len) + i + 1 : kv_len", "(kv_len - q_len) + i : kv_len", None),
    ("causal_top_left", "(kv_len - q_len) + i + 1 : kv_len", "i + 1 : kv_len", None),
    ("pv_reads_k", "out[e] += w * elem(v_buffer", "out[e] += w * elem(k_buffer", None),
    ("layer_offset_dropped_k",
     "int64_t k_off = (((int64_t)layer_id * size + slot) * n_kv_heads + g) * head_dim;",
     "int64_t k_off = (((int64_t)slot) * n_kv_heads + g) * head_dim;", None),
    ("no_normalisation", "out[e] /= denom;", "out[e] /= 1.0;", None),
    ("q_row_transposed", "int64_t row = (int64_t)b * n_heads + h;",
     "int64_t row = (int64_t)h * batch + b;", None),
    ("prefill_request_lookup", "while (qo_indptr[b + 1] <= p)", "while (qo_indptr[b + 1] < p)", None),
    ("bf16_widening", "<< 16", "<< 8", None),
    ("kv_write_layer", "int64_t dst = ((int64_t)layer_id * size + loc) * row;",
     "int64_t dst = ((int64_t)loc) * row;", None),
    ("rope_sign", "out[base + 2 * i] = re * c - im * s;", "out[base + 2 * i] = re * c + im * s;", None),
    ("rope_cos_sin_swapped", "double c = cs[2 * i], s = cs[2 * i + 1];",
     "double c = cs[2 * i + 1], s = cs[2 * i];", None),
]


def _mutate(text, old, new, which):
    assert old in text, f"mutation anchor vanished from the oracle source: {old!r}"
    if which is None:
        return text.replace(old, new)
    start = -1
    for _ in range(which + 1):
        start = text.index(old, start + 1)
    return text[:start] + new + text[start + len(old):]


def _run_pins(so_path):
    env = dict(os.environ, PKV_ORACLE_SO=so_path)
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           PINS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


@pytest.mark.parametrize("name,old,new,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new, which):
    text = open(SRC).read()
    src = tmp_path / "mutant.c"
    src.write_text(_mutate(text, old, new, which))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-o", str(so), str(src), "-lm"])
    r = _run_pins(str(so))
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
