"""Pins for the scheduling oracle (oracle/plan_oracle.py) against the worked
examples the pages print (tests/golden/plan_examples.json) and against
invariants of the split partition."""
import json
import os

import numpy as np
import pytest

from oracle import plan_oracle as po

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_examples.json")


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_num_splits_worked_example(golden):
    for ex in golden["num_splits"]:
        sms, tiles = ex["num_sms"], ex["total_mblocks"]
        # K long enough to split, one m block per tile, small KV head (no L2 branch)
        for max_splits in (3, 16, 128):
            s = po.num_splits_heuristic(tiles, sms, 64, 1, 1 << 20, False, max_splits)
            assert s == ex["expect_splits"]
        for k, eff in ex["efficiency_by_splits"].items():
            w = tiles * int(k) / sms
            assert round(w / np.ceil(w), 2) == pytest.approx(eff, abs=0.005)


def test_num_splits_gates():
    # grid already fills >= 0.8 of the SMs and the KV head fits the L2 budget -> 1
    assert po.num_splits_heuristic(130, 148, 1024, 1, 1 << 20, False, 128) == 1
    # filled grid, huge KV head, many m blocks, not causal -> ceil(size / 50 MB)
    size = 3 * po.L2_SPLIT_BYTES + 1
    assert po.num_splits_heuristic(400, 148, 4096, 400, size, False, 128) == 4
    assert po.num_splits_heuristic(400, 148, 4096, 400, size, True, 128) == 1
    # short K: at most 4 n blocks -> 1
    assert po.num_splits_heuristic(4, 148, 4, 1, 1 << 20, False, 128) == 1


def test_pack_gqa_worked_example(golden):
    for ex in golden["pack_gqa"]:
        assert po.should_pack_gqa(False, ex["seqlen_q"], ex["qhead_per_khead"], ex["block_m"]) \
            == ex["expect_pack"]
        assert ex["seqlen_q"] / 128 == pytest.approx(ex["nopack_efficiency"], abs=5e-4)
    assert po.should_pack_gqa(True, 8192, 1, 128) is True
    assert po.should_pack_gqa(False, 8192, 4, 128) is False
    assert po.should_pack_gqa(False, 1, 8, 128) is True


def test_causal_block_skip_worked_example(golden):
    for ex in golden["causal_skip"]:
        n, bm, bn = ex["seqlen"], ex["block_m"], ex["block_n"]
        nm = n // bm
        total = 0
        for m in range(nm):
            lo, hi = po.n_block_min_max(n, n, m, bm, bn, True, False, -1, 0, False, 1)
            total += hi - lo
        assert total == ex["computed_blocks"]
        assert nm * po.ceil_div(n, bn) == ex["total_blocks"]


def test_fixed_chunk_nsplit_worked_example(golden):
    for ex in golden["nsplit_fixed_chunk"]:
        s = po.nsplit_fixed_chunk(ex["kv_len"])
        assert s == ex["expect_nsplit"]
        assert ex["base_blocks"] * s == ex["expect_grid_blocks"]
    assert po.nsplit_fixed_chunk(1) == 1
    assert po.nsplit_fixed_chunk(10 ** 7) == 32


def test_block_bounds_agree_with_element_mask(oracle_mod):
    """The block-level bounds (section 3.2) must cover exactly the blocks that
    hold a visible key under the oracle's element-level mask."""
    rng = np.random.default_rng(3)
    for _ in range(60):
        sq = int(rng.integers(1, 300))
        sk = int(rng.integers(1, 700))
        bm = int(rng.choice([16, 64, 128]))
        bn = int(rng.choice([64, 128]))
        causal = bool(rng.integers(0, 2))
        wl = int(rng.choice([-1, 0, 5, 100]))
        local = wl >= 0
        wr = 0 if causal else 1 << 30
        # element-level truth from the oracle's rule, by one-hot probing counts
        for m in range((sq + bm - 1) // bm):
            rows = range(m * bm, min(sq, (m + 1) * bm))
            need = set()
            for i in rows:
                diag = i + sk - sq
                for j in range(sk):
                    if causal and j > diag:
                        continue
                    if local and j < diag - wl:
                        continue
                    need.add(j // bn)
            lo, hi = po.n_block_min_max(sq, sk, m, bm, bn, causal or local, local,
                                        max(wl, 0), wr if local else 0, False, 1)
            if not causal and local:
                lo, hi = po.n_block_min_max(sq, sk, m, bm, bn, False, True, wl, 1 << 30, False, 1)
            if need:
                assert lo <= min(need) and max(need) < hi, (sq, sk, bm, bn, causal, wl, m)
                # no fully masked block at either end
                assert lo == min(need) or not local
                assert hi - 1 == max(need)
    # the oracle's element mask counts agree with the brute-force loop above
    assert oracle_mod.count_visible(37, 50, 1, 4) == sum(
        1 for i in range(37) for j in range(50) if i + 13 - 4 <= j <= i + 13)


def test_split_partition_tiles_the_range():
    rng = np.random.default_rng(5)
    for _ in range(500):
        sq = int(rng.integers(1, 64))
        sk = int(rng.integers(0, 5000))
        S = int(rng.integers(1, 40))
        lo0, hi0 = po.n_block_min_max(sq, sk, 0, 64, 128, False, False, -1, 0, True, 4)
        covered = []
        for t in range(S):
            lo, hi = po.n_block_min_max(sq, sk, 0, 64, 128, False, False, -1, 0, True, 4,
                                        split_word=(S << 16) | t)
            covered.extend(range(lo, hi))
        assert covered == list(range(lo0, hi0))


def test_split_counts_cover_each_sequence():
    rng = np.random.default_rng(6)
    for _ in range(200):
        B = int(rng.integers(1, 33))
        lens = [int(x) for x in rng.integers(0, 70000, size=B)]
        S = int(rng.integers(1, 130))
        counts = po.split_counts(lens, 128, S)
        nmax = max(po.ceil_div(n, 128) for n in lens)
        for n, c in zip(lens, counts):
            nb = po.ceil_div(n, 128)
            assert 1 <= c <= max(S, 1)
            if S > 1 and nmax > 0:
                chunk = po.ceil_div(nmax, S)
                assert (c - 1) * chunk < max(nb, 1) <= c * chunk or nb == 0
