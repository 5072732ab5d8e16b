"""The product's host scheduler (libskattn.so, sk_attn_plan / sk_attn_plan_ranges)
against the scheduling oracle written from the pages: packing decision, split
counts of the page-derived policies, per-sequence split counts and the KV block
range of every CTA must match bit for bit.  The GPU echo test then checks that
the kernels use exactly these ranges.

An empty block range has no unique representation (the printed block formulas
leave (min, max) with min >= max in several forms; the product reports [0, 0)),
so for a range the oracle finds empty the product's range must be empty too,
and every other field is compared exactly."""
import numpy as np
import pytest

from oracle import plan_oracle as po
import workloads as wl


@pytest.fixture(scope="module")
def sk():
    from split_kv_flash_gb300 import build as b
    b.build()
    import split_kv_flash_gb300 as sk
    return sk


POLICIES = {"fa": 2, "fixed_chunk": 3, "min_chunk": 4}


def same_table(got, exp):
    """Per-CTA tables agree: words and work flags exactly, non-empty ranges
    exactly, empty ranges as empty."""
    if len(got) != len(exp):
        return False
    for g, e in zip(got, exp):
        if g[2] != e[2] or g[3] != e[3]:
            return False
        if e[1] > e[0]:
            if (g[0], g[1]) != (e[0], e[1]):
                return False
        elif g[1] > g[0]:
            return False
    return True


def _opts(sk, policy=0, num_sms=148, **kw):
    o = sk.Opts()
    o.policy = policy
    o.num_sms = num_sms
    for k, v in kw.items():
        setattr(o, k, v)
    return o


def _expected(sk, info, B, Hq, Hkv, sq, kv, d, causal, window, policy, num_sms, force_splits=0):
    G = Hq // Hkv
    pack = po.should_pack_gqa(False, sq, G, 128) and G > 1
    assert bool(info.pack_gqa) == pack
    head_tiles = Hkv if pack else Hq
    assert info.head_tiles == head_tiles
    rows = sq * (G if pack else 1)
    assert info.rows_per_head_tile == rows
    nm = po.ceil_div(rows, info.kBlockM) if rows else 0
    assert info.num_m_blocks == nm
    if force_splits:
        S = min(force_splits, 128, max(po.ceil_div(max(kv), 128), 1))
    else:
        S = po.choose_splits(policy, B, head_tiles, nm, kv, d, 128, num_sms, causal or window >= 0)
    assert info.num_splits_policy == S
    sb = po.split_counts(kv, 128, S)
    assert info.num_splits == max(sb)
    return po.cta_table(sq, kv, G, pack, head_tiles, info.kBlockM, 128, nm, info.num_splits, sb,
                        causal, window)


def _cases():
    rng = np.random.default_rng(1234)
    cases = [
        # the workloads' shapes
        (1, 4, 4, 1, [256], 64, False, -1),
        (1, 32, 4, 1, [4096], 128, False, -1),
        (1, 32, 4, 1, [131072], 128, False, -1),
        (2, 16, 16, 9, [128 + 9] * 2, 128, True, -1),
        (2, 16, 16, 33, [8192 + 33] * 2, 128, True, -1),
        (4, 32, 8, 1, wl.varlen_lengths(4, 1302), 128, False, -1),
        (32, 32, 8, 1, wl.varlen_lengths(32, 1305), 128, False, -1),
        (4, 32, 8, 8192, [8192] * 4, 128, True, -1),
        (4, 32, 8, 8192, [8192] * 4, 128, True, 1024),
        # edge cases: ragged, empty sequences, window without causal, sk < sq
        (3, 8, 2, 5, [0, 1, 300], 64, True, -1),
        (2, 12, 3, 40, [17, 1000], 128, False, 50),
        (1, 2, 1, 200, [150], 128, True, 7),
        (1, 64, 8, 2, [999], 64, True, 0),
        # whole tiles that see no key (q_len far above kv_len, causal)
        (1, 4, 4, 1000, [10], 128, True, -1),
        (2, 8, 2, 700, [0, 50], 64, True, 30),
        (3, 16, 2, 900, [0, 1, 2], 128, True, 0),
    ]
    for _ in range(60):
        B = int(rng.integers(1, 9))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 4, 8]))
        sq = int(rng.choice([1, 2, 5, 9, 17, 33, 64, 100, 300]))
        if rng.random() < 0.5:
            kv = [int(rng.integers(0, 5000))] * B
        else:
            kv = [int(x) for x in rng.integers(0, 9000, size=B)]
        causal = bool(rng.integers(0, 2))
        window = int(rng.choice([-1, -1, 0, 33, 1024]))
        cases.append((B, Hkv * G, Hkv, sq, kv, int(rng.choice([64, 128])), causal, window))
    return cases


@pytest.mark.parametrize("policy", sorted(POLICIES))
def test_plan_matches_oracle(sk, policy):
    for num_sms in (108, 148, 152):
        for (B, Hq, Hkv, sq, kv, d, causal, window) in _cases():
            o = _opts(sk, POLICIES[policy], num_sms)
            info = sk.sk_attn_plan(B, Hq, Hkv, sq, kv, d, causal, window, o)
            exp = _expected(sk, info, B, Hq, Hkv, sq, kv, d, causal, window, policy, num_sms)
            got = sk.sk_attn_plan_ranges(B, Hq, Hkv, sq, kv, d, causal, window, o)
            assert same_table(got, exp), (B, Hq, Hkv, sq, kv, d, causal, window, policy, num_sms)


def test_forced_split_counts_match_oracle(sk):
    for S in (1, 2, 3, 7, 40, 128, 500):
        for (B, Hq, Hkv, sq, kv, d, causal, window) in _cases()[:20]:
            o = _opts(sk, 0, 148, force_num_splits=S)
            info = sk.sk_attn_plan(B, Hq, Hkv, sq, kv, d, causal, window, o)
            exp = _expected(sk, info, B, Hq, Hkv, sq, kv, d, causal, window, None, 148, S)
            got = sk.sk_attn_plan_ranges(B, Hq, Hkv, sq, kv, d, causal, window, o)
            assert same_table(got, exp)


def test_fill_policy_invariants(sk):
    """The default policy (own, measured choice): splits tile each range exactly,
    every CTA fits in one wave when splitting (unless sequences of different
    lengths on the decode path chose a multi-wave count by list schedule), and no
    split repeats a chunk."""
    for num_sms in (148, 152):
        for (B, Hq, Hkv, sq, kv, d, causal, window) in _cases():
            o = _opts(sk, 0, num_sms)
            info = sk.sk_attn_plan(B, Hq, Hkv, sq, kv, d, causal, window, o)
            S = info.num_splits_policy
            sb = po.split_counts(kv, 128, S)
            assert info.num_splits == max(sb)
            if info.needs_combine:
                ctas = sum(c * info.head_tiles * info.num_m_blocks for c in sb)
                if ctas > num_sms:
                    assert B > 1 and len(set(kv)) > 1 and info.path == sk.SK_PATH_DECODE
                    assert S in (2, 4, 8, 16)
                if info.path == sk.SK_PATH_DECODE:
                    # a split pays for the combine only when it saves 3 blocks
                    nblk = po.ceil_div(max(kv), 128)
                    assert nblk - po.ceil_div(nblk, S) >= 3
            G = Hq // Hkv
            pack = bool(info.pack_gqa)
            exp = po.cta_table(sq, kv, G, pack, info.head_tiles, info.kBlockM, 128,
                               info.num_m_blocks, info.num_splits, sb, causal, window)
            assert same_table(sk.sk_attn_plan_ranges(B, Hq, Hkv, sq, kv, d, causal, window, o), exp)


def test_short_verify_keeps_one_split(sk):
    """Speculative verify (B=2, 16 heads, causal): over 137 or 265 keys the
    decode path takes one split (the combine would cost more than the blocks
    it saves); over 2057 keys it splits."""
    for kv, split in ((137, False), (265, False), (2057, True)):
        info = sk.sk_attn_plan(2, 16, 16, 9, [kv] * 2, 128, True, -1, _opts(sk, 0, 152))
        assert info.path == sk.SK_PATH_DECODE
        assert bool(info.needs_combine) == split, kv


def _list_schedule(table, sms, overhead=4.0, empty=0.3):
    """Finishing time (in KV blocks) of the CTAs of a plan table taken in launch
    order by the first free SM."""
    import heapq
    free = [0.0] * sms
    end = 0.0
    for lo, hi, _word, work in table:
        t = heapq.heappop(free)
        t += (hi - lo + overhead) if work else empty
        end = max(end, t)
        heapq.heappush(free, t)
    return end


def test_varlen_decode_split_count_by_list_schedule(sk):
    """Decode of 16 sequences of different lengths on 152 SMs: one wave (the
    fill policy gives one split) leaves the longest sequences streaming alone,
    so the planner takes a multi-wave split count, the one among 1, 2, 4, 8, 16
    whose list schedule (recomputed here from the oracle's per-CTA ranges)
    finishes first, by more than 3 % where it differs from one split."""
    import workloads as wl
    w = wl.varlen_decode(16)
    info = sk.sk_attn_plan(w.B, w.Hq, w.Hkv, 1, w.kv_len, 128, opts=_opts(sk, 0, 152))
    S = info.num_splits_policy
    assert S > 1 and info.num_ctas > 152
    G = w.Hq // w.Hkv
    times = {}
    for c in (1, 2, 4, 8, 16):
        sb = po.split_counts(w.kv_len, 128, c)
        table = po.cta_table(1, w.kv_len, G, bool(info.pack_gqa), info.head_tiles, info.kBlockM, 128,
                             info.num_m_blocks, max(sb), sb, False, -1)
        times[c] = _list_schedule(table, 152)
    assert times[S] <= min(times.values()) / 0.97 + 1e-9
    assert times[S] < 0.97 * times[1]
    # equal lengths keep one wave
    info = sk.sk_attn_plan(4, 32, 8, 1, [20000] * 4, 128, opts=_opts(sk, 0, 152))
    assert info.num_ctas <= 152


def test_gqa_decode_split_counts(sk):
    """GQA decode at 131072 keys: the section 5.2 heuristic gives 32 splits on
    148 SMs (4 tiles); the default policy fills all 152 SMs of a GB300."""
    info = sk.sk_attn_plan(1, 32, 4, 1, [131072], 128, opts=_opts(sk, POLICIES["fa"], 148))
    assert info.num_splits_policy == 32
    info = sk.sk_attn_plan(1, 32, 4, 1, [131072], 128, opts=_opts(sk, 0, 152))
    assert info.num_splits == 38 and info.num_ctas == 152
    assert info.path == sk.SK_PATH_DECODE and info.kBlockM == 16 and info.pack_gqa == 1


def test_product_ranges_match_brute_force_visibility(sk):
    """The product's block ranges against the definition of visibility,
    independently of the scheduling oracle: a tile's range is exactly the KV
    blocks holding a key that some row of the tile sees, and the splits of a
    tile cut that range into consecutive shares of ceil(range / splits)."""
    rng = np.random.default_rng(77)
    for _ in range(150):
        G = int(rng.choice([1, 2, 4, 8]))
        Hkv = 1
        sq = int(rng.choice([1, 2, 3, 9, 17, 33, 64, 100, 300]))
        sk_len = int(rng.integers(0, 1200))
        causal = bool(rng.integers(0, 2))
        wl = int(rng.choice([-1, -1, 0, 5, 130, 700]))
        S = int(rng.integers(1, 6))
        o = _opts(sk, 0, 148, force_num_splits=S)
        if rng.random() < 0.3:
            o.force_path = sk.SK_PATH_PREFILL
        info = sk.sk_attn_plan(1, Hkv * G, Hkv, sq, [sk_len], 128, causal, wl, o)
        table = sk.sk_attn_plan_ranges(1, Hkv * G, Hkv, sq, [sk_len], 128, causal, wl, o)
        g = G if info.pack_gqa else 1
        rows, bm, nm, ns = info.rows_per_head_tile, info.kBlockM, info.num_m_blocks, info.num_splits
        masked = causal or wl >= 0
        for bx in range(nm):
            m = nm - 1 - bx if masked else bx
            need = set()
            for r in range(m * bm, min((m + 1) * bm, rows)):
                diag = r // g + sk_len - sq
                lo_key = max(0, diag - wl) if wl >= 0 else 0
                hi_key = min(sk_len - 1, diag) if causal else sk_len - 1
                need.update(range(lo_key // 128, hi_key // 128 + 1) if hi_key >= lo_key else [])
            covered = []
            for s in range(ns):
                lo, hi, word, work = table[s * nm + bx]  # head tile 0
                assert work == 1 and word == (ns << 16) | s
                covered.extend(range(lo, hi))
            assert covered == sorted(need), (G, sq, sk_len, causal, wl, S, m)
            if need:
                share = -(-len(need) // ns)
                assert all(table[s * nm + bx][1] - table[s * nm + bx][0] <= share for s in range(ns))


def test_packed_tile_map_matches_oracle(sk):
    """The packed tile map (tiling chapter section 4.5): on the decode path,
    when sequences of one batch have different split counts, the grid is one
    dimension over exactly the CTAs with work, in the oracle's packed launch
    order; everywhere else the option leaves the rectangular grid."""
    packed_seen = 0
    for num_sms in (148, 152):
        for (B, Hq, Hkv, sq, kv, d, causal, window) in _cases():
            o = _opts(sk, 0, num_sms, tile_map=sk.SK_TILE_MAP_PACKED)
            info = sk.sk_attn_plan(B, Hq, Hkv, sq, kv, d, causal, window, o)
            sb = po.split_counts(kv, 128, info.num_splits_policy)
            work = sum(sb) * info.head_tiles * info.num_m_blocks
            grid = info.head_tiles * info.num_splits * info.num_m_blocks * B
            packed = info.path == sk.SK_PATH_DECODE and B > 1 and work < grid
            assert info.tile_map == (sk.SK_TILE_MAP_PACKED if packed else sk.SK_TILE_MAP_GRID)
            exp = po.cta_table(sq, kv, Hq // Hkv, bool(info.pack_gqa), info.head_tiles, info.kBlockM, 128,
                               info.num_m_blocks, info.num_splits, sb, causal, window, packed=packed)
            got = sk.sk_attn_plan_ranges(B, Hq, Hkv, sq, kv, d, causal, window, o)
            assert same_table(got, exp), (B, Hq, Hkv, sq, kv, d, causal, window, num_sms)
            if packed:
                packed_seen += 1
                assert (info.grid_x, info.grid_y, info.grid_z) == (work, 1, 1)
                assert info.num_ctas == work
                # the same problem without the option: the grid, and the same tiles
                g = sk.sk_attn_plan(B, Hq, Hkv, sq, kv, d, causal, window, _opts(sk, 0, num_sms))
                assert g.tile_map == sk.SK_TILE_MAP_GRID and g.num_ctas == grid
                full = sk.sk_attn_plan_ranges(B, Hq, Hkv, sq, kv, d, causal, window, _opts(sk, 0, num_sms))
                assert [list(r) for r in full if r[3]] == [list(r) for r in got]
    assert packed_seen >= 10


def test_unknown_tile_map_is_rejected(sk):
    with pytest.raises(sk.SKError) as ei:
        sk.sk_attn_plan(2, 8, 2, 1, [100, 5000], 128, False, -1, _opts(sk, tile_map=3))
    assert ei.value.status == 1
