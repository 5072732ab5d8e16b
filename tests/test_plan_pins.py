"""Pins for the composed scheduling oracle (oracle/plan_oracle.py: mask_flags,
choose_splits, nsplit_min_chunk, split_counts, cta_table).

Two kinds of pin, neither computed by code under test:
  * hand-enumerated tables (tests/golden/plan_tables.json), each entry citing
    the passage it follows and showing its arithmetic;
  * brute force from the definition of visibility (query i sees key j when
    j <= i + kv_len - q_len under a causal mask and j >= i + kv_len - q_len -
    window_left under a left window): a tile's KV block range must be exactly
    the blocks that hold a key some row of the tile sees.

Every pin takes the oracle module as an argument, so that
tests/test_oracle_mutations.py can run the same pins against copies of the
module with planted mistakes.
"""
import json
import os

import numpy as np

from oracle import plan_oracle as _po

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_tables.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def pin_cta_tables(po):
    for t in _golden()["cta_tables"]:
        got = po.cta_table(**t["args"])
        assert [list(x) for x in got] == t["expect"], t["name"]


def pin_split_counts(po):
    for t in _golden()["split_counts"]:
        assert po.split_counts(t["kv_lens"], t["block_n"], t["num_splits"]) == t["expect"]


def pin_min_chunk(po):
    for t in _golden()["min_chunk"]:
        got = po.nsplit_min_chunk(t["num_sms"], t["tiles"], t["kv_len"], min_chunk=t["min_chunk"],
                                  blocks_per_sm=t["blocks_per_sm"])
        assert got == t["expect_splits"], t["reasoning"]
        if "unfloored_chunk" in t:
            # the review's figure: keys per split when every SM runs blocks_per_sm CTAs
            per_head = t["blocks_per_sm"] * t["num_sms"] // t["tiles"]
            assert round(t["kv_len"] / per_head) == t["unfloored_chunk"]
            assert got * t["min_chunk"] == t["kv_len"]


def pin_choose_splits(po):
    for t in _golden()["choose_splits"]:
        got = po.choose_splits(t["policy"], t["B"], t["head_tiles"], t["num_m_blocks"], t["kv_lens"],
                               t["d"], t["block_n"], t["num_sms"], t["causal_or_local"],
                               t.get("max_splits_opt", 128))
        assert got == t["expect"], t["cite"]


def pin_mask_flags(po):
    for row in _golden()["mask_flags"][0]["table"]:
        exp = list(row["expect"])
        if exp[3] == "open":
            got = po.mask_flags(row["causal"], row["window_left"])
            assert list(got[:3]) == exp[:3]
            assert got[3] >= 1 << 29, "a window without causal leaves the right side open"
        else:
            assert list(po.mask_flags(row["causal"], row["window_left"])) == exp


def _visible_blocks(sq, sk, rows_lo, rows_hi, G, causal, wl, bn):
    """Blocks holding a key that some packed row in [rows_lo, rows_hi) sees, by
    enumeration of the definition."""
    blocks = set()
    for r in range(rows_lo, rows_hi):
        i = r // G
        diag = i + sk - sq
        for j in range(sk):
            if causal and j > diag:
                continue
            if wl >= 0 and j < diag - wl:
                continue
            blocks.add(j // bn)
    return blocks


def pin_tiles_match_visibility(po, n_cases=120, seed=11):
    rng = np.random.default_rng(seed)
    for _ in range(n_cases):
        G = int(rng.choice([1, 2, 3, 4]))
        pack = G > 1 and bool(rng.integers(0, 2))
        sq = int(rng.integers(1, 40))
        sk = int(rng.integers(0, 90))
        bm = int(rng.choice([8, 16, 32]))
        bn = int(rng.choice([8, 16]))
        causal = bool(rng.integers(0, 2))
        wl = int(rng.choice([-1, -1, 0, 3, 17]))
        rows = sq * (G if pack else 1)
        nm = -(-rows // bm)
        masked = causal or wl >= 0
        S = int(rng.integers(1, 5))
        table = po.cta_table(sq, [sk], G, pack, 1, bm, bn, nm, S, [S], causal, wl)
        assert len(table) == nm * S
        for bx in range(nm):
            m = nm - 1 - bx if masked else bx
            need = _visible_blocks(sq, sk, m * bm, min((m + 1) * bm, rows), G if pack else 1, causal, wl, bn)
            full = (min(need), max(need) + 1) if need else None
            got = [table[s * nm + bx] for s in range(S)]
            covered = []
            for s, (lo, hi, word, work) in enumerate(got):
                assert word == (S << 16) | s and work == 1
                covered.extend(range(lo, hi))
            if full is None:
                assert covered == [], (sq, sk, G, pack, bm, bn, causal, wl, m)
                continue
            assert covered == list(range(*full)), (sq, sk, G, pack, bm, bn, causal, wl, m, got, full)
            share = -(-(full[1] - full[0]) // S)
            for lo, hi, _, _ in got:
                assert hi - lo <= share


PINS = [pin_cta_tables, pin_split_counts, pin_min_chunk, pin_choose_splits, pin_mask_flags,
        pin_tiles_match_visibility]


def test_cta_tables_hand_enumerated():
    pin_cta_tables(_po)


def test_split_counts_hand_enumerated():
    pin_split_counts(_po)


def test_min_chunk_review_example():
    pin_min_chunk(_po)


def test_choose_splits_hand_computed():
    pin_choose_splits(_po)


def test_mask_flags_truth_table():
    pin_mask_flags(_po)


def test_tiles_match_brute_force_visibility():
    pin_tiles_match_visibility(_po)
