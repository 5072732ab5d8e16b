"""The oracle pins must catch plausible mistakes.

Each case plants one mistake in a private copy of oracle/attn_oracle.c (on the
CPU, in a temporary directory), builds it, and runs the pins of
test_oracle_pins.py against the mutated library: at least one pin must fail.
"""
import ctypes
import inspect
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild
import tests.test_oracle_pins as pins

MUTATIONS = {
    "gqa_head_map_modulo": ("const long hk = h / G;", "const long hk = h % Hkv;"),
    "causal_offset_dropped": ("long diag = i + sk - sq;", "long diag = i;"),
    "window_bound_exclusive": ("if (wl >= 0 && j < diag - wl) return 0;",
                               "if (wl >= 0 && j <= diag - wl) return 0;"),
    "scale_dropped": ("double x = scale * dot;", "double x = dot;"),
    "max_not_subtracted": ("sum += exp(x - mx);", "sum += exp(x);"),
    "weights_not_normalised": ("double w = exp(x - lse);", "double w = exp(x - mx);"),
    "value_used_as_key": ("const uint16_t* krow = k +", "const uint16_t* krow = v +"),
    "bf16_widening_shift": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "merge_weight_wrong": ("double w = exp(l_part[t] - total);", "double w = exp(l_part[t] - mx);"),
    "merge_lse_drops_max": ("total = mx + log(acc);", "total = log(acc);"),
}

PIN_TESTS = [(n, f) for n, f in inspect.getmembers(pins, inspect.isfunction) if n.startswith("test_")]


def _build_mutant(tmp_path, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, old
    path = tmp_path / "attn_oracle.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(path), "-o",
                    str(lib), "-lm"], check=True)
    return str(lib)


def _run_pins():
    failed = []
    for name, fn in PIN_TESTS:
        params = inspect.signature(fn).parameters
        marks = getattr(fn, "pytestmark", [])
        arg_sets = [{}]
        for m in marks:
            if m.name == "parametrize":
                names = [s.strip() for s in m.args[0].split(",")]
                arg_sets = [dict(zip(names, v if isinstance(v, tuple) else (v,))) for v in m.args[1]]
        for args in arg_sets:
            kwargs = dict(args)
            if "oracle_mod" in params:
                kwargs["oracle_mod"] = oracle
            try:
                fn(**kwargs)
            except Exception:  # noqa: BLE001 - any failure counts as caught
                failed.append(name)
                break
    return failed


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, mutation):
    old, new = MUTATIONS[mutation]
    lib_path = _build_mutant(tmp_path, old, new)
    real = oracle.lib()
    mutant = ctypes.CDLL(lib_path)
    for fname in ("oracle_attn_rows", "oracle_attn_fwd", "oracle_attn_fwd_split",
                  "oracle_count_visible"):
        getattr(mutant, fname).argtypes = getattr(real, fname).argtypes
        getattr(mutant, fname).restype = getattr(real, fname).restype
    oracle._lib = mutant
    try:
        failed = _run_pins()
    finally:
        oracle._lib = real
    assert failed, "no pin caught mutation %s" % mutation


def test_unmutated_oracle_passes_every_pin():
    """Control: the same runner reports no failure on the real oracle."""
    assert _run_pins() == []
