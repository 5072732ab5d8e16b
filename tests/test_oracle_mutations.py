"""The oracle pins must catch plausible mistakes.

Each case plants one mistake in a private copy of oracle/attn_oracle.c (on the
CPU, in a temporary directory), builds it, and runs the pins of
test_oracle_pins.py against the mutated library: at least one pin must fail.
The same is done for the scheduling oracle (oracle/plan_oracle.py): a copy of
its source with one planted mistake is loaded as a separate module and the pins
of test_plan_pins.py and test_plan_oracle.py run against it.
"""
import ctypes
import inspect
import json
import os
import subprocess
import types

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
    "value_rows_at_key_stride": ("const uint16_t* vrow = v + (((size_t)(off + j)) * Hkv + hk) * (size_t)dv;",
                                 "const uint16_t* vrow = v + (((size_t)(off + j)) * Hkv + hk) * (size_t)d;"),
    "value_width_truncated": ("for (int c = 0; c < dv; ++c) o_row[c] += w * bf16_bits_to_double(vrow[c]);",
                              "for (int c = 0; c < d && c < dv; ++c) o_row[c] += w * bf16_bits_to_double(vrow[c]);"),
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
                  "oracle_count_visible", "oracle_attn_rows_v", "oracle_attn_fwd_v"):
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


# ------------------------------------------------------------ scheduling oracle
PLAN_MUTATIONS = {
    "lpt_order_off": ("reverse = bool(causal) or window_left >= 0", "reverse = False"),
    "causal_window_right_open": ("0 if causal else WINDOW_RIGHT_OPEN)", "WINDOW_RIGHT_OPEN)"),
    "max_splits_not_clipped_to_blocks":
        ("max_splits = max(1, min(min(max_splits_opt, MAX_SPLITS), max(nblk_max, 1)))",
         "max_splits = max(1, min(max_splits_opt, MAX_SPLITS))"),
    "kv_head_bytes_k_only": ("max_kv * 2 * d * 2", "max_kv * d * 2"),
    "min_chunk_takes_max": ("return max(1, min(fill, by_chunk))", "return max(1, max(fill, by_chunk))"),
    "min_chunk_fill_floor": ("fill = ceil_div(blocks_per_sm * num_sms, tiles)",
                             "fill = (blocks_per_sm * num_sms) // tiles"),
    "split_chunk_floor": ("chunk = ceil_div(nmax, num_splits)", "chunk = max(1, nmax // num_splits)"),
    "split_word_swapped": ("word = (sb << 16) | split", "word = (split << 16) | sb"),
    "packed_rows_not_converted": ("m_idx_max = c_div(m_idx_max - 1, qhead_per_khead) + 1",
                                  "m_idx_max = m_idx_max"),
    "local_lower_bound_dropped": ("n_block_min = max(0, c_div(n_idx_left, block_n))", "n_block_min = 0"),
    "block_offset_dropped": ("n_idx = m_idx_max + seqlen_k - seqlen_q", "n_idx = m_idx_max"),
    "packed_keeps_empty_ctas": ("                    if not packed:\n", "                    if True:\n"),
    "heuristic_threshold_080": (">= 0.85 * float(best)", ">= 0.8 * float(best)"),
    "l2_budget_32mb": ("L2_SPLIT_BYTES = 50 * 1024 * 1024", "L2_SPLIT_BYTES = 32 * 1024 * 1024"),
    "split_share_floor": ("per = ceil_div(n_block_max - n_block_min, n_split)",
                          "per = max(1, (n_block_max - n_block_min) // n_split)"),
}


def _plan_mutant(old, new):
    from oracle import plan_oracle
    src = open(plan_oracle.__file__).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("plan_oracle_mutant")
    mod.__file__ = "<mutant>"
    exec(compile(src.replace(old, new), "<plan_oracle_mutant>", "exec"), mod.__dict__)
    return mod


def _run_plan_pins(mod):
    import tests.test_plan_oracle as tpo
    import tests.test_plan_pins as tpp
    failed = []
    for pin in tpp.PINS:
        try:
            pin(mod)
        except Exception:  # noqa: BLE001 - any failure counts as caught
            failed.append(pin.__name__)
    with open(tpo.GOLDEN) as f:
        golden = json.load(f)
    saved = tpo.po
    tpo.po = mod
    try:
        for name, fn in inspect.getmembers(tpo, inspect.isfunction):
            if not name.startswith("test_"):
                continue
            params = inspect.signature(fn).parameters
            kwargs = {}
            if "golden" in params:
                kwargs["golden"] = golden
            if "oracle_mod" in params:
                kwargs["oracle_mod"] = oracle
            try:
                fn(**kwargs)
            except Exception:  # noqa: BLE001
                failed.append(name)
    finally:
        tpo.po = saved
    return failed


@pytest.mark.parametrize("mutation", sorted(PLAN_MUTATIONS))
def test_planted_plan_mistake_is_caught(mutation):
    old, new = PLAN_MUTATIONS[mutation]
    assert _run_plan_pins(_plan_mutant(old, new)), "no pin caught mutation %s" % mutation


def test_unmutated_plan_oracle_passes_every_pin():
    from oracle import plan_oracle
    assert _run_plan_pins(plan_oracle) == []
