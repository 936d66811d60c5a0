"""Pins of the CPU oracle against what the pages and plain mathematics fix.

Nothing here re-types the oracle's formulas: the expected values are the
pages' printed examples (``tests/golden``), independent formulations (numpy's
own C-order layout for the coordinate map, concatenated block lists for the
range formula, numpy fancy indexing for copies) and invariants (round trips,
untouched bytes, the null block).
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_39_gb300 import workloads as wl

BITS = oracle.ERR_BITS


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- slot map


def test_figure6_paged(golden):
    g = golden("figure6_bs4.json")
    T = g["block_size"]
    for step in g["steps"]:
        row = np.zeros((1, 8), np.int32)
        row[0, :len(step["row"])] = step["row"]
        pos = np.array(step["positions"], np.int64)
        n = len(pos)
        slots, err = oracle.slot_mapping_paged([0, n], pos, row, n, n, T, 16)
        assert err == 0
        assert slots.tolist() == step["slots"], step["what"]


def test_figure6_range(golden):
    g = golden("figure6_bs4.json")
    T = g["block_size"]
    runs = g["ranges_final_row"]
    rs = np.zeros((1, 256), np.int32)
    rl = np.zeros((1, 256), np.int32)
    for i, (s, ln) in enumerate(runs):
        rs[0, i], rl[0, i] = s, ln
    all_pos = np.concatenate([np.array(s["positions"], np.int64) for s in g["steps"]])
    all_slots = sum((s["slots"] for s in g["steps"]), [])
    n = len(all_pos)
    slots, err = oracle.slot_mapping_range([0, n], all_pos, rs, rl, [len(runs)], n, n, T, 16)
    assert err == 0
    assert slots.tolist() == all_slots


def test_page3_block16(golden):
    g = golden("page3_bs16.json")
    T = g["block_size"]
    row = np.zeros((1, 8), np.int32)
    row[0, :2] = g["row"]
    pos = np.array(g["positions"], np.int64)
    n = len(pos)
    slots, err = oracle.slot_mapping_paged([0, n], pos, row, n, n, T, 16)
    assert err == 0
    for k, v in g["checked"].items():
        assert slots[int(k)] == v
    assert slots[:16].tolist() == list(range(112, 128))


def test_tail_is_pad():
    row = np.array([[3, 4]], np.int32)
    slots, err = oracle.slot_mapping_paged([0, 3], [0, 1, 17], row, 3, 11, 16, 8)
    assert err == 0
    assert slots.tolist() == [48, 49, 65] + [-1] * 8


def test_null_entries_and_padding_rows_are_pad():
    # request 0 owns [5, 0(null), 6]; rows 1..3 are CUDA-graph padding rows
    table = np.zeros((4, 8), np.int32)
    table[0, :3] = [5, 0, 6]
    pos = np.array([0, 15, 16, 31, 32, 40], np.int64)
    qsl = [0, 6, 6, 6, 6]
    slots, err = oracle.slot_mapping_paged(qsl, pos, table, 6, 9, 16, 8)
    assert err == 0
    assert slots.tolist() == [80, 95, -1, -1, 96, 104, -1, -1, -1]


def test_position_beyond_table_is_pad():
    table = np.array([[1, 2]], np.int32)
    slots, err = oracle.slot_mapping_paged([0, 2], [31, 32], table, 2, 2, 16, 4)
    assert err == 0
    assert slots.tolist() == [47, -1]


def test_negative_position_and_bad_block_flagged():
    table = np.array([[1, 7, -3]], np.int32)
    slots, err = oracle.slot_mapping_paged([0, 4], [-1, 0, 16, 32], table, 4, 4, 16, 4)
    assert slots.tolist() == [-1, 16, -1, -1]
    assert err == BITS["BAD_POSITION"] | BITS["BAD_BLOCK"]


def test_bad_qsl_flagged():
    table = np.array([[1], [2]], np.int32)
    _, err = oracle.slot_mapping_paged([0, 3, 2], [0, 1, 2], table, 3, 3, 16, 4)
    assert err & BITS["BAD_QSL"]
    _, err = oracle.slot_mapping_paged([0, 1, 5], [0, 1, 2], table, 3, 3, 16, 4)
    assert err & BITS["BAD_QSL"]


def test_tokens_outside_every_span_are_pad():
    table = np.array([[1]], np.int32)
    slots, err = oracle.slot_mapping_paged([1, 2], [0, 0, 0], table, 3, 3, 16, 4)
    assert err == 0
    assert slots.tolist() == [-1, 16, -1]


def _brute_range_slot(p, starts, lens, T, B):
    """Independent formulation: the request's logical block list is the
    concatenation of its ranges; logical block lb is element lb of it."""
    if p < 0:
        return -1
    blocks = []
    for s, ln in zip(starts, lens):
        blocks.extend(range(int(s), int(s) + max(int(ln), 0)))
    lb = p // T
    if lb >= len(blocks):
        return -1
    b = blocks[lb]
    if b == 0 or b < 0 or b >= B:
        return -1
    return b * T + p % T


@pytest.mark.parametrize("seed", range(12))
def test_range_matches_concatenated_block_lists(seed):
    rng = _rng(100 + seed)
    T = int(rng.choice([1, 4, 16]))
    B = 40
    R = 5
    S = 8
    rs = rng.integers(-2, B + 3, size=(R, S)).astype(np.int32)
    rl = rng.integers(-1, 5, size=(R, S)).astype(np.int32)
    nr = rng.integers(0, S + 1, size=R).astype(np.int32)
    lens = rng.integers(0, 6, size=R)
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(qsl[-1])
    pos = rng.integers(-1, 30 * T, size=N).astype(np.int64)
    slots, err = oracle.slot_mapping_range(qsl, pos, rs, rl, nr, N, N + 2, T, B)
    exp_err = 0
    for r in range(R):
        if any(rl[r, i] <= 0 for i in range(nr[r])):
            exp_err |= BITS["BAD_RANGE"]
        for t in range(qsl[r], qsl[r + 1]):
            e = _brute_range_slot(int(pos[t]), rs[r, :nr[r]], rl[r, :nr[r]], T, B)
            assert slots[t] == e
            if pos[t] < 0:
                exp_err |= BITS["BAD_POSITION"]
            else:
                blocks = [b for s, ln in zip(rs[r, :nr[r]], rl[r, :nr[r]])
                          for b in range(int(s), int(s) + max(int(ln), 0))]
                lb = int(pos[t]) // T
                if lb < len(blocks) and (blocks[lb] < 0 or blocks[lb] >= B):
                    exp_err |= BITS["BAD_BLOCK"]
    assert slots[N:].tolist() == [-1, -1]
    assert err == exp_err


def test_range_descriptor_count_over_stride_is_bad_range():
    rs = np.array([[1, 5]], np.int32)
    rl = np.array([[1, 1]], np.int32)
    slots, err = oracle.slot_mapping_range([0, 1], [0], rs, rl, [3], 1, 1, 16, 8)
    assert slots.tolist() == [-1]
    assert err == BITS["BAD_RANGE"]


def test_zero_length_range_is_bad_range_and_covers_nothing():
    rs = np.array([[4, 9, 2]], np.int32)
    rl = np.array([[1, 0, 2]], np.int32)
    slots, err = oracle.slot_mapping_range([0, 3], [0, 16, 40], rs, rl, [3], 3, 3, 16, 16)
    assert err == BITS["BAD_RANGE"]
    assert slots.tolist() == [64, 32, 56]


def test_range_cap_fails_closed():
    rs = np.zeros((1, 257), np.int32)
    with pytest.raises(oracle.OracleError) as ei:
        oracle.slot_mapping_range([0, 0], [], rs, rs, [0], 0, 0, 16, 8)
    assert ei.value.status == oracle.EUNSUPPORTED


def _concat_blocks(starts, lens):
    out = []
    for s_, ln in zip(starts, lens):
        out.extend(range(int(s_), int(s_) + max(int(ln), 0)))
    return out


@pytest.mark.parametrize("seed", range(8))
def test_table_from_ranges_matches_concatenation(seed):
    rng = _rng(200 + seed)
    R, S, stride = 4, 6, 12
    rs = rng.integers(1, 50, size=(R, S)).astype(np.int32)
    rl = rng.integers(-1, 4, size=(R, S)).astype(np.int32)
    nr = rng.integers(0, S + 1, size=R).astype(np.int32)
    if seed % 3 == 0:
        nr[0] = S + 1  # malformed row
    table, err = oracle.table_from_ranges(rs, rl, nr, stride, with_error=True)
    exp_err = 0
    for r in range(R):
        if nr[r] > S:
            exp_err |= BITS["BAD_RANGE"]
            assert (table[r] == 0).all()
            continue
        if (rl[r, :nr[r]] <= 0).any():
            exp_err |= BITS["BAD_RANGE"]
        blocks = _concat_blocks(rs[r, :nr[r]], rl[r, :nr[r]])
        if len(blocks) > stride:
            exp_err |= BITS["OUT_OF_SPACE"]
        blocks = blocks[:stride]
        assert table[r].tolist() == blocks + [0] * (stride - len(blocks))
    assert err == exp_err


def test_table_from_ranges_zero_length_and_cut_rows():
    """A range of length 0 covers nothing and marks its row malformed; ranges
    reaching past the table row are cut at its end.  Each case alone, so each
    error bit is pinned on its own."""
    rs = np.array([[5, 20, 9]], np.int32)
    rl = np.array([[3, 0, 2]], np.int32)
    table, err = oracle.table_from_ranges(rs, rl, [3], 8, with_error=True)
    assert table.tolist() == [[5, 6, 7, 9, 10, 0, 0, 0]]
    assert err == BITS["BAD_RANGE"]
    rs = np.array([[1, 30]], np.int32)
    rl = np.array([[4, 6]], np.int32)
    table, err = oracle.table_from_ranges(rs, rl, [2], 8, with_error=True)
    assert table.tolist() == [[1, 2, 3, 4, 30, 31, 32, 33]]
    assert err == BITS["OUT_OF_SPACE"]
    table, err = oracle.table_from_ranges(rs, rl, [2], 10, with_error=True)
    assert table.tolist() == [[1, 2, 3, 4, 30, 31, 32, 33, 34, 35]] and err == 0


@pytest.mark.parametrize("name", ["tiny", "decode", "mixed"])
def test_range_equals_paged_on_expanded_table(name):
    """Range and table strategies give identical slots for the same layout."""
    w = wl.CONFIGS[name]()
    for key, lay in w.layouts.items():
        if lay.range_start is None:
            continue
        table, terr = oracle.table_from_ranges(lay.range_start, lay.range_len, lay.num_ranges,
                                               lay.table_stride, with_error=True)
        assert terr == 0
        assert np.array_equal(table, lay.table), key
        a, ea = oracle.slot_mapping_paged(w.qsl, w.positions, table, w.num_tokens,
                                          w.max_num_tokens, w.block_size, w.num_blocks)
        b, eb = oracle.slot_mapping_range(w.qsl, w.positions, lay.range_start, lay.range_len,
                                          lay.num_ranges, w.num_tokens, w.max_num_tokens,
                                          w.block_size, w.num_blocks)
        assert ea == eb == 0
        assert np.array_equal(a, b)
        assert (a[:w.num_tokens] >= w.block_size).all()  # never the null block
        assert (a[w.num_tokens:] == -1).all()


def test_paged_slots_unique_and_in_owned_blocks():
    w = wl.tiny()
    lay = w.layouts["P"]
    slots, err = oracle.slot_mapping_paged(w.qsl, w.positions, lay.table, w.num_tokens,
                                           w.max_num_tokens, w.block_size, w.num_blocks)
    assert err == 0
    real = slots[:w.num_tokens]
    assert len(set(real.tolist())) == len(real)
    for r in range(w.num_reqs):
        owned = set(lay.table[r][lay.table[r] > 0].tolist())
        for t in range(w.qsl[r], w.qsl[r + 1]):
            assert real[t] // w.block_size in owned
            assert real[t] % w.block_size == w.positions[t] % w.block_size


# ------------------------------------- context-parallel filter (unpinned)
# The filter's formula is not on the pages (the listing is cut off): only the
# world-size-1 case and the stated properties (real slots for the rank's own
# tokens, PAD elsewhere; every token on exactly one rank) are pinned.


@pytest.mark.parametrize("seed", range(6))
def test_cp_world_size_one_is_the_paged_map(seed):
    rng = _rng(800 + seed)
    T = int(rng.choice([4, 16]))
    table = rng.integers(-1, 40, size=(3, 8)).astype(np.int32)
    lens = rng.integers(0, 30, size=3)
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(qsl[-1])
    pos = rng.integers(-1, 9 * T, size=N).astype(np.int64)
    a, ea = oracle.slot_mapping_paged(qsl, pos, table, N, N + 3, T, 40)
    for I in (1, 2, T):
        b, eb = oracle.slot_mapping_paged_cp(qsl, pos, table, N, N + 3, T, 40, 1, 0, I)
        assert eb == ea and np.array_equal(a, b)


@pytest.mark.parametrize("W,I,T", [(2, 1, 16), (4, 1, 16), (4, 4, 16), (8, 2, 16), (2, 16, 16),
                                   (3, 2, 4)])
def test_cp_partition_and_balance(W, I, T):
    rng = _rng(900 + W * 10 + I)
    stride = 6
    table = rng.permutation(np.arange(1, 100))[:2 * stride].reshape(2, stride).astype(np.int32)
    n = stride * T * W
    qsl = np.array([0, n, 2 * n], np.int32)
    pos = np.concatenate([np.arange(n), np.arange(n)]).astype(np.int64)
    per_rank = []
    for k in range(W):
        s_, e_ = oracle.slot_mapping_paged_cp(qsl, pos, table, 2 * n, 2 * n, T, 100, W, k, I)
        assert e_ == 0
        per_rank.append(s_)
    owned = np.stack([s_ >= 0 for s_ in per_rank])
    assert (owned.sum(axis=0) == 1).all()          # every token on exactly one rank
    for k, s_ in enumerate(per_rank):
        mine = s_[s_ >= 0]
        assert len(np.unique(mine)) == len(mine)    # distinct slots per rank
        t_idx = np.nonzero(s_ >= 0)[0]
        r_idx = (t_idx >= n).astype(int)
        lb = pos[t_idx] // (T * W)
        assert np.array_equal(mine // T, table[r_idx, lb])   # in the entry's block
        # balance: each virtual block gives each rank exactly T tokens, offsets 0..T-1
        for r in range(2):
            for j in range(stride):
                sel = (r_idx == r) & (lb == j)
                assert sorted((mine[sel] % T).tolist()) == list(range(T))


def test_cp_rejects_bad_arguments():
    args = ([0, 1], [0], np.array([[1]], np.int32), 1, 1, 16, 4)
    with pytest.raises(oracle.OracleError) as ei:
        oracle.slot_mapping_paged_cp(*args, 2, 0, 3)   # interleave does not divide block size
    assert ei.value.status == oracle.EUNSUPPORTED
    for W, k, I in ((0, 0, 1), (2, 2, 1), (2, -1, 1), (2, 0, 0)):
        with pytest.raises(oracle.OracleError) as ei:
            oracle.slot_mapping_paged_cp(*args, W, k, I)
        assert ei.value.status == oracle.EINVAL


# ------------------------------------------------------------ coordinates


def test_coord_is_c_order_layout_of_l_b_t():
    L, B, T = 3, 7, 5
    ids = np.arange(L * B * T).reshape(L, B, T)
    for l in range(L):
        for b in range(B):
            for t in range(T):
                assert oracle.coord(l, b, t, B, T) == ids[l, b, t]


def test_coord_64bit_page_layout():
    # the page's coordinate layout: 32 layers x 64K blocks x 32 tokens/block x 2048 B/token
    L, B, T, bpt = 32, 65536, 32, 2048
    n = oracle.coord(L - 1, B - 1, T - 1, B, T)
    assert n == L * B * T - 1
    assert n * bpt == L * B * T * bpt - bpt > 2 ** 32


# ------------------------------------------------------------------ write


def _cache(shape, seed):
    return _rng(seed).integers(0, 2 ** 16, size=shape, dtype=np.uint16)


def test_write_matches_numpy_5d_indexing():
    rng = _rng(7)
    L, B, T, H, D, N = 3, 9, 4, 2, 8, 11
    slots = rng.permutation(np.arange(T, B * T))[:N].astype(np.int64)
    slots[[2, 5]] = -1
    key = _cache((L, N, H, D), 1)
    val = _cache((L, N, H, D), 2)
    kc = _cache((L, B, T, H, D), 3)
    vc = _cache((L, B, T, H, D), 4)
    ek, ev = kc.copy(), vc.copy()
    for t in range(N):
        if slots[t] < 0:
            continue
        b, o = divmod(int(slots[t]), T)
        ek[:, b, o] = key[:, t]
        ev[:, b, o] = val[:, t]
    err = oracle.cache_write(key, val, kc, vc, slots, B, T)
    assert err == 0
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_write_skips_null_block_and_out_of_range_slots():
    L, B, T, H, D = 2, 4, 4, 1, 8
    key = _cache((L, 4, H, D), 5)
    kc = _cache((L, B, T, H, D), 6)
    vc = _cache((L, B, T, H, D), 7)
    before_k, before_v = kc.copy(), vc.copy()
    slots = np.array([-1, 2, B * T, 5], np.int64)  # PAD, null block, past end, valid
    err = oracle.cache_write(key, key, kc, vc, slots, B, T)
    assert err == BITS["NULL_WRITE"] | BITS["BAD_SLOT"]
    assert np.array_equal(kc[:, 0], before_k[:, 0])  # null block untouched
    changed = np.argwhere((kc != before_k).any(axis=(3, 4)))
    assert sorted(map(tuple, changed.tolist())) == [(0, 1, 1), (1, 1, 1)]
    assert np.array_equal(kc[:, 1, 1], key[:, 3])


def test_write_rows_agree_with_full_write():
    w = wl.tiny()
    lay = w.layouts["G"]
    slots, _ = oracle.slot_mapping_paged(w.qsl, w.positions, lay.table, w.num_tokens,
                                         w.max_num_tokens, w.block_size, w.num_blocks)
    rows, err = oracle.write_rows(slots[:w.num_tokens], w.num_tokens, 2, w.num_blocks, w.block_size)
    assert err == 0
    E = 16
    key = _cache((2, w.num_tokens, 2, 8), 8)
    kc = np.zeros((2, w.num_blocks, w.block_size, 2, 8), np.uint16)
    oracle.cache_write(key, key, kc, kc.copy(), slots[:w.num_tokens], w.num_blocks, w.block_size)
    flat = kc.reshape(-1, E)
    for l in range(2):
        for t in range(w.num_tokens):
            assert np.array_equal(flat[rows[l, t]], key[l, t].reshape(E))


# ----------------------------------------------------------------- gather


def _write_then_gather(w, lay, seed, layer=0, L=1):
    H, D = 2, 8
    slots, err = oracle.slot_mapping_paged(w.qsl, w.positions, lay.table, w.num_tokens,
                                           w.max_num_tokens, w.block_size, w.num_blocks)
    assert err == 0
    key = _cache((L, w.num_tokens, H, D), seed)
    val = _cache((L, w.num_tokens, H, D), seed + 1)
    kc = _cache((L, w.num_blocks, w.block_size, H, D), seed + 2)
    vc = _cache((L, w.num_blocks, w.block_size, H, D), seed + 3)
    assert oracle.cache_write(key, val, kc, vc, slots[:w.num_tokens], w.num_blocks,
                              w.block_size) == 0
    rows = int((w.gather_end - w.gather_start).sum())
    ko = np.zeros((rows, H, D), np.uint16)
    vo = np.zeros((rows, H, D), np.uint16)
    err = oracle.cache_gather(kc, vc, layer, w.num_blocks, w.block_size, lay.table,
                              w.gather_start, w.gather_end, ko, vo)
    return key, val, ko, vo, err


@pytest.mark.parametrize("layout", ["P", "G"])
def test_gather_after_write_is_identity(layout):
    w = wl.tiny()
    key, val, ko, vo, err = _write_then_gather(w, w.layouts[layout], 11, layer=1, L=2)
    assert err == 0
    # tiny prompts start at position 0, so the gather returns the tokens in order
    assert np.array_equal(ko, key[1]) and np.array_equal(vo, val[1])


def test_gather_contiguous_range_is_one_memcpy():
    T, H, D, B = 4, 2, 8, 30
    s = 9
    table = np.zeros((2, 8), np.int32)
    table[0, :5] = np.arange(s, s + 5)
    table[1, :3] = np.arange(20, 23)
    kc = _cache((1, B, T, H, D), 12)
    vc = _cache((1, B, T, H, D), 13)
    g0, g1 = np.array([3, 1], np.int32), np.array([19, 12], np.int32)
    rows = int((g1 - g0).sum())
    ko = np.zeros((rows, H, D), np.uint16)
    vo = np.zeros((rows, H, D), np.uint16)
    assert oracle.cache_gather(kc, vc, 0, B, T, table, g0, g1, ko, vo) == 0
    flat_k = kc.reshape(-1, H, D)
    assert np.array_equal(ko[:16], flat_k[s * T + 3: s * T + 19])
    assert np.array_equal(ko[16:], flat_k[20 * T + 1: 20 * T + 12])
    assert np.array_equal(vo[16:], vc.reshape(-1, H, D)[20 * T + 1: 20 * T + 12])


def test_gather_null_entries_are_zero_rows_and_errors():
    T, H, D, B = 4, 1, 8, 6
    table = np.array([[2, 0, 9, 3]], np.int32)
    kc = _cache((1, B, T, H, D), 14)
    ko = np.full((16, H, D), 7, np.uint16)
    vo = ko.copy()
    err = oracle.cache_gather(kc, kc, 0, B, T, table, [0], [16], ko, vo)
    assert err == BITS["BAD_BLOCK"]
    assert (ko[4:12] == 0).all()
    assert np.array_equal(ko[:4], kc[0, 2]) and np.array_equal(ko[12:], kc[0, 3])


def test_gather_out_of_space_and_bad_spans():
    T, H, D, B = 4, 1, 8, 6
    table = np.array([[1, 2], [3, 4]], np.int32)
    kc = _cache((1, B, T, H, D), 15)
    ko = np.full((5, H, D), 7, np.uint16)
    vo = ko.copy()
    err = oracle.cache_gather(kc, kc, 0, B, T, table, [0, 5], [6, 2], ko, vo)
    assert err == BITS["OUT_OF_SPACE"] | BITS["BAD_POSITION"]
    assert np.array_equal(ko[:4], kc[0, 1]) and np.array_equal(ko[4], kc[0, 2, 0])
    # rows past out_rows are neither resolved nor written
    src, err2 = oracle.gather_rows(0, B, T, table, [0, 0], [3, 9], 8)
    assert err2 == BITS["OUT_OF_SPACE"]
    assert src.tolist() == [4, 5, 6, 12, 13, 14, 15, 16]
    # a position past the table row is a zero row with BAD_POSITION
    src, err3 = oracle.gather_rows(0, B, T, table, [0, 0], [3, 9], 13)
    assert err3 == BITS["BAD_POSITION"]
    assert src.tolist() == [4, 5, 6, 12, 13, 14, 15, 16, 17, 18, 19, -1, -2]


# ------------------------------------------------- range-addressed gather


@pytest.mark.parametrize("seed", range(10))
def test_gather_range_matches_concatenated_blocks(seed):
    """Source rows of the range gather: logical block lb of request r is element
    lb of its concatenated ranges; the row index is numpy's own C-order index
    of (layer, block, offset) in a [L, B, T] grid."""
    rng = _rng(600 + seed)
    T, B, L, R, S = int(rng.choice([1, 4, 16])), 60, 3, 5, 6
    layer = int(rng.integers(0, L))
    rs = rng.integers(-1, B + 2, size=(R, S)).astype(np.int32)
    rl = rng.integers(-1, 5, size=(R, S)).astype(np.int32)
    nr = rng.integers(0, S + 1, size=R).astype(np.int32)
    if seed % 4 == 0:
        nr[1] = S + 2
    g0 = rng.integers(-1, 10 * T, size=R).astype(np.int32)
    g1 = (g0 + rng.integers(-2, 12 * T, size=R)).astype(np.int32)
    total = int(np.where((g0 >= 0) & (g1 >= g0), g1 - g0, 0).sum())
    out_rows = total - (seed % 3)
    src, err = oracle.gather_rows_range(layer, B, T, rs, rl, nr, g0, g1, max(out_rows, 0))
    exp_err, o_r = 0, 0
    exp = np.full(max(out_rows, 0), -2, np.int64)
    for r in range(R):
        if nr[r] > S or (rl[r, :max(nr[r], 0)] <= 0).any():
            exp_err |= BITS["BAD_RANGE"]
    for r in range(R):
        if g0[r] < 0 or g1[r] < g0[r]:
            exp_err |= BITS["BAD_POSITION"]
            continue
        blocks = _concat_blocks(rs[r, :nr[r]], rl[r, :nr[r]]) if nr[r] <= S else []
        for p in range(int(g0[r]), int(g1[r])):
            o = o_r + p - int(g0[r])
            if o >= out_rows:
                exp_err |= BITS["OUT_OF_SPACE"]
                continue
            lb = p // T
            exp[o] = -1
            if lb < len(blocks):
                b = blocks[lb]
                if b < 0 or b >= B:
                    exp_err |= BITS["BAD_BLOCK"]
                elif b != 0:
                    exp[o] = np.ravel_multi_index((layer, b, p % T), (L, B, T))
        o_r += int(g1[r]) - int(g0[r])
    assert err == exp_err
    assert np.array_equal(src, exp)


@pytest.mark.parametrize("name", ["tiny", "decode", "long"])
def test_gather_range_equals_table_gather(name):
    w = wl.CONFIGS[name]()
    lay = w.layouts["G"]
    rows = int((w.gather_end.astype(np.int64) - w.gather_start).sum())
    a, ea = oracle.gather_rows(0, w.num_blocks, w.block_size, lay.table, w.gather_start,
                               w.gather_end, rows)
    b, eb = oracle.gather_rows_range(0, w.num_blocks, w.block_size, lay.range_start, lay.range_len,
                                     lay.num_ranges, w.gather_start, w.gather_end, rows)
    assert ea == eb == 0
    assert np.array_equal(a, b)


# ---------------------------------------------------------- copy-on-write


def test_copy_blocks_matches_slice_assignment():
    rng = _rng(700)
    L, B, T, H, D = 3, 20, 4, 2, 8
    kc = _cache((L, B, T, H, D), 70)
    vc = _cache((L, B, T, H, D), 71)
    src = np.array([3, 5, 0, 7, 9, 2, 4], np.int32)
    dst = np.array([11, 12, 13, 0, 25, 14, 15], np.int32)
    ek, ev = kc.copy(), vc.copy()
    for a_, b_ in zip(src, dst):
        if 0 < a_ < B and 0 < b_ < B:
            ek[:, b_] = ek[:, a_]
            ev[:, b_] = ev[:, a_]
    err = oracle.copy_blocks(kc, vc, src, dst)
    assert err == BITS["BAD_BLOCK"] | BITS["NULL_WRITE"]
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)
    assert np.array_equal(kc[:, 0], _cache((L, B, T, H, D), 70)[:, 0])  # null block kept


def test_copy_blocks_then_write_diverges_only_the_copy():
    """Copy-on-write: after copying a shared block and writing into the copy,
    the original block is unchanged and the copy differs in one row."""
    L, B, T, H, D = 2, 10, 4, 1, 8
    kc = _cache((L, B, T, H, D), 72)
    vc = _cache((L, B, T, H, D), 73)
    orig = kc.copy()
    assert oracle.copy_blocks(kc, vc, [4], [8]) == 0
    key = _cache((L, 1, H, D), 74)
    assert oracle.cache_write(key, key, kc, vc, np.array([8 * T + 2], np.int64), B, T) == 0
    assert np.array_equal(kc[:, 4], orig[:, 4])
    diff = (kc[:, 8] != orig[:, 4]).any(axis=(2, 3))
    assert diff.tolist() == [[False, False, True, False]] * L


# ----------------------------------------------------------------- expand


def test_expand_golden(golden):
    g = golden("expand_32_16.json")
    out, err = oracle.expand_kernel_blocks(np.array([g["mgr_row"]], np.int32),
                                           g["mgr_block_size"], g["kernel_block_size"])
    assert err == 0
    assert out[0].tolist() == g["kernel_row"]
    for mbs, kbs in g["rejected"]:
        with pytest.raises(oracle.OracleError) as ei:
            oracle.expand_kernel_blocks(np.array([[1]], np.int32), mbs, kbs, 4)
        assert ei.value.status == oracle.EUNSUPPORTED


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_expand_matches_repeat_formulation(k):
    rng = _rng(300 + k)
    mgr = rng.integers(0, 1000, size=(5, 7)).astype(np.int32)
    mgr[rng.random(mgr.shape) < 0.3] = 0
    out, err = oracle.expand_kernel_blocks(mgr, 16 * k, 16, 7 * k + 3)
    assert err == 0
    rep = np.repeat(mgr.astype(np.int64), k, axis=1) * k + np.tile(np.arange(k), 7)
    rep[np.repeat(mgr, k, axis=1) == 0] = 0
    assert np.array_equal(out[:, :7 * k], rep)
    assert (out[:, 7 * k:] == 0).all()
    if k == 1:
        assert np.array_equal(out[:, :7], mgr)


def test_expand_overflow_and_negative_flagged():
    mgr = np.array([[2 ** 30, -4, 3]], np.int32)
    out, err = oracle.expand_kernel_blocks(mgr, 32, 16)
    assert err == BITS["BAD_BLOCK"]
    assert out[0].tolist() == [0, 0, 0, 0, 6, 7]


def test_expand_then_slot_map_matches_manager_slots():
    """A manager-level slot and the kernel-level slot of the expanded table
    address the same token: slot_kernel == slot_manager for the same cache."""
    rng = _rng(17)
    mgr = rng.permutation(np.arange(1, 40))[:16].reshape(2, 8).astype(np.int32)
    kt, _ = oracle.expand_kernel_blocks(mgr, 32, 16)
    pos = rng.integers(0, 8 * 32, size=20).astype(np.int64)
    qsl = [0, 10, 20]
    sm, e1 = oracle.slot_mapping_paged(qsl, pos, mgr, 20, 20, 32, 40)
    sk, e2 = oracle.slot_mapping_paged(qsl, pos, kt, 20, 20, 16, 80)
    assert e1 == e2 == 0
    assert np.array_equal(sm, sk)


# ------------------------------------------------- workload structure pins


def test_swa_recycling_example(golden):
    g = golden("swa_recycling.json")
    n = wl.swa_null_prefix(g["num_computed"], g["window"], g["block_size"])
    assert n == g["null_blocks"]
    assert n * g["block_size"] == g["printed_freed_tokens_roughly"]


def test_table_stride_alignment():
    assert wl.table_stride_for(3, 16) == 8
    assert wl.table_stride_for(256, 16) == 256
    assert wl.table_stride_for(1024, 32) == 1024
    assert wl.table_stride_for(1, 128) == 1


def test_range_stride_for():
    # the run cap rounded up to 16-byte rows, never past the backend's cap
    assert [wl.range_stride_for(m) for m in (1, 3, 4, 5, 8, 16, 255, 256, 300)] == \
        [4, 4, 4, 8, 8, 16, 256, 256, 256]


@pytest.mark.parametrize("name,cap", [("tiny", 3), ("decode", 4), ("mixed", 8), ("long", 16)])
def test_descriptor_rows_sized_to_the_run_cap(name, cap):
    """Layout G's descriptor rows hold the layout's run cap (rounded up to a
    multiple of 4), and every request's ranges fit; layout P keeps 256."""
    w = wl.CONFIGS[name]()
    g = w.layouts["G"]
    assert g.range_start.shape[1] == g.range_len.shape[1] == wl.range_stride_for(cap)
    assert 1 <= g.num_ranges[g.num_ranges > 0].min() and g.num_ranges.max() <= cap
    if "P" in w.layouts and w.layouts["P"].range_start is not None:
        assert w.layouts["P"].range_start.shape[1] == wl.RANGE_CAP


@pytest.mark.parametrize("name", ["tiny", "decode", "mixed", "long"])
def test_workload_structure(name):
    w = wl.CONFIGS[name]()
    assert w.qsl[0] == 0 and w.qsl[-1] == w.num_tokens
    assert (np.diff(w.qsl) >= 0).all()
    for lay in w.layouts.values():
        used = lay.table[lay.table > 0]
        assert len(np.unique(used)) == len(used)  # no physical block shared
        assert used.max() < w.num_blocks
        assert (lay.table >= 0).all()
        if lay.num_ranges is not None:
            assert lay.num_ranges.max() <= wl.RANGE_CAP
    assert w.positions.dtype == np.int64


def test_hybrid_structure():
    h = wl.hybrid()
    assert h.num_reqs == 640 and h.num_real_reqs == 512
    assert (np.diff(h.qsl[512:]) == 0).all()
    for g in h.groups.values():
        assert (g.mgr_table[512:] == 0).all()
        used = g.mgr_table[g.mgr_table > 0]
        assert len(np.unique(used)) == len(used)
        assert used.max() < g.mgr_num_blocks
    swa = h.groups["swa"]
    for r in range(0, 512, 37):
        c = int(h.ctx[r])
        nnull = wl.swa_null_prefix(c - 1, h.window, 32)
        assert (swa.mgr_table[r, :nnull] == 0).all()
        assert (swa.mgr_table[r, nnull:-(-c // 32)] > 0).all()
        # the window's positions never fall into a recycled block
        assert swa.gather_start[r] // 32 >= nnull
