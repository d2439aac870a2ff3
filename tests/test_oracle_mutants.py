"""The oracle's pins must be strong enough to catch plausible slips.

Each case copies attn_oracle.cpp to a temporary directory, plants one mistake
in the copy (the oracle itself is never modified), builds it with g++, swaps it
in for the real library and checks that at least one pin of
tests/test_oracle.py fails.  CPU only.
"""

import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.cpp")

MUTANTS = {
    "scale dropped": ("score[j] = dot * scale;", "score[j] = dot;"),
    "key index transposed": ("K.at(b, h, j, e)", "K.at(b, h, i, e)"),
    "value row mismatched": ("o_row[e] += a * V.at(b, h, j, e);", "o_row[e] += a * V.at(b, h, i, e);"),
    "no max subtraction in sum": ("d += std::exp(s[i] - m);", "d += std::exp(s[i]);"),
    "merge sign flipped": ("d = d * f_old + d_blk * std::exp(m_blk - m_new);",
                           "d = d * f_old + d_blk * std::exp(m_new - m_blk);"),
    "history not rescaled": ("d = d * f_old + d_blk", "d = d + d_blk"),
    "lse uses log10": ("*lse = m + std::log(l);", "*lse = m + std::log10(l);"),
    "layout strides swapped": ("*sh = d;\n    *ss = rs;", "*sh = rs;\n    *ss = d;"),
    "split: head from wrong index": ("head = (c % D) / d, e = c % d;", "head = (c % d) % H, e = c % d;"),
    "f16 exponent bias off": ("expo - 15", "expo - 14"),
    # (mutants must keep every index in bounds: they run inside the test process)
    "grouped: group stride too small": ("(h / hg) * S * hg * d + s * hg * d", "(h / hg) * S * d + s * hg * d"),
    "projection transposed weight": ("wd[i] = load_elem(w, et, i);",
                                     "wd[i] = load_elem(w, et, (i % N) * D + i / N);"),
}

PIN_FUNCS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _run_pins():
    """Number of pins that fail (parametrised pins run with a few fixed arguments)."""
    fails = 0
    for f in PIN_FUNCS:
        marks = getattr(f, "pytestmark", [])
        arg_sets = [()]
        for m in marks:
            if m.name == "parametrize":
                arg_sets = [a if isinstance(a, tuple) else (a,) for a in m.args[1]]
        for args in arg_sets:
            try:
                f(*args)
            except Exception:
                fails += 1
    return fails


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for '{name}' not found"
    mut = tmp_path / "mut.cpp"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(mut), "-o", str(so)],
                   check=True)
    saved = oracle._load()
    oracle._lib = oracle.bind(ctypes.CDLL(str(so)))
    try:
        assert _run_pins() > 0, f"no pin caught the planted mistake: {name}"
    finally:
        oracle._lib = saved


def test_unmutated_oracle_passes_all_pins():
    assert _run_pins() == 0
