"""The oracle pins must fail for plausible mistakes planted in the oracle.

Each mutant is a copy of the oracle's C source with one line changed, built
into a temporary library on the CPU. The pins of test_oracle.py run against it
and at least one of them must fail.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild

import test_oracle as T

MUTANTS = {
    "kv head by modulo": ("const int g = h / group;", "const int g = h % jb->kv.hkv;"),
    "sink scaled": ("const double sink = has_sink ? (double)jb->sinks[h] : -INFINITY;",
                    "const double sink = has_sink ? (double)jb->sinks[h] * jb->scale : -INFINITY;"),
    "sink left out of denominator": ("double den = has_sink ? exp(sink - z) : 0.0;",
                                     "double den = 0.0;"),
    "window one key too wide": ("(long)j <= p - jb->window", "(long)j < p - jb->window"),
    "top-left causal alignment": ("const long p = (long)(lk - lq) + i;", "const long p = i;"),
    "lse without sink": ("*lse = z + log(den);",
                         "*lse = z + log(den - (has_sink ? exp(sink - z) : 0.0));"),
    "merge drops the sink": ("double wsum = sinks ? exp((double)sinks[h] - m) : 0.0;",
                             "double wsum = 0.0;"),
    "score sign flipped": ("s[n] = jb->scale * dot;", "s[n] = -jb->scale * dot;"),
}


def _build_mutant(tmp_path, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", str(path),
                    "-o", str(lib), "-lm"], check=True)
    return str(lib)


def _pins_pass(oracle_mod):
    checks = [
        lambda: [T.test_oracle_matches_decimal_brute_force(oracle_mod, s) for s in T.TINY],
        lambda: T.test_oracle_closed_forms(oracle_mod),
        lambda: [T.test_oracle_split_blocks_merge_to_whole(oracle_mod, n) for n in (2, 3)],
        lambda: [T.test_oracle_sink_scales_plain_attention(oracle_mod, w) for w in (0, 6)],
    ]
    for chk in checks:
        try:
            chk()
        except AssertionError:
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name, monkeypatch):
    old, new = MUTANTS[name]
    path = _build_mutant(tmp_path, old, new)
    monkeypatch.setattr(obuild, "build", lambda force=False: path)
    monkeypatch.setattr(oracle, "_LIB", None)
    try:
        assert not _pins_pass(oracle), "pins did not catch: " + name
    finally:
        oracle._LIB = None


def test_unmutated_oracle_passes_the_same_checks(oracle_lib):
    assert _pins_pass(oracle_lib)
