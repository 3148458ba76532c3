"""Pins of the oracle's worklist by brute force on tiny packs.

"03 · 长文负载均衡" §3.2: a computation block exists only for a (Q block,
KV block) pair whose mask is not all zero, and a tile is charged its exact
query-key pair count.  These tests rebuild, element by element, the pairs
each worklist unit would compute (slice semantics: FULL, or CAUSAL on
positions with an optional window) and check them against the mask predicate
written from the definitions: every allowed pair is computed exactly once per
head and no tile in a run is empty.
"""
import itertools

import numpy as np
import pytest

from packed_varlen_attention_cu_gb300 import workloads as W


def slice_accepts(sl, i, j, smask=None):
    q_row0, q_len, q_pos0, k_row0, k_len, k_pos0, typ, win = (int(x) for x in sl)
    if not (q_row0 <= i < q_row0 + q_len and k_row0 <= j < k_row0 + k_len):
        return False
    if typ == 0:
        return True
    qp, kp = q_pos0 + i - q_row0, k_pos0 + j - k_row0
    if typ == 4:  # packed: the row's own document (rows that start one are flagged)
        starts = [r for r in range(q_len) if (int(smask[r // 32]) >> (r % 32)) & 1]
        if max(st for st in starts if st <= qp) > kp:
            return False
    return kp <= qp and (win <= 0 or qp - kp < win)


def coverage(wl, tq, tk, hq, tile_m, tile_n):
    cov = np.zeros((hq, tq, tk), dtype=np.int32)
    per_unit = []
    empty_tiles = 0
    for u in wl["units"]:
        uid, seg, t0, t1, h0, h1, kvh, rb, rc, cta = (int(x) for x in u)
        sg = wl["segs"][seg]
        subs = [(t0, h0)] + ([(t1, h1)] if h1 >= 0 else [])
        cnt = 0
        for r in range(rb, rb + rc):
            sidx, lo, hi = (int(x) for x in wl["runs"][r])
            sl = wl["slices"][sidx]
            sm = wl["slice_masks"][sidx] if "slice_masks" in wl else None
            assert sl[0] == sg[0] and sl[1] == sg[1]
            for kt in range(lo, hi):
                k0 = sl[3] + kt * tile_n
                k1 = min(k0 + tile_n, sl[3] + sl[4])
                hit = 0
                for (t, h) in subs:
                    r0 = sg[0] + t * tile_m
                    r1 = min(r0 + tile_m, sg[0] + sg[1])
                    for i in range(r0, r1):
                        for j in range(k0, k1):
                            if slice_accepts(sl, i, j, sm):
                                cov[h, i, j] += 1
                                cnt += 1
                                hit += 1
                empty_tiles += hit == 0
        per_unit.append(cnt)
    return cov, np.array(per_unit), empty_tiles


CASES = [
    ([5, 17, 1, 9, 0, 12], W.MASK_CAUSAL, {}),
    ([23, 3, 16], W.MASK_SLIDING_WINDOW, {"window": 5}),
    ([16, 7, 9, 13], W.MASK_SHARED_QUESTION, {"num_prefix": 1}),
    ([6, 5, 11, 4], W.MASK_SHARED_QUESTION, {"num_prefix": 2}),
]


@pytest.mark.parametrize("lengths,kind,kw", CASES)
@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (3, 1), (2, 1)])
@pytest.mark.parametrize("tile_m,tile_n", [(4, 4), (8, 4), (4, 8)])
def test_worklist_covers_allowed_pairs_once(oracle_mod, lengths, kind, kw, hq, hkv, tile_m, tile_n):
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    m = oracle_mod.Mask(kind, **kw)
    wl = oracle_mod.worklist(cu, m, tile_m, tile_n, hq, hkv, num_ctas=5, c_tile=3)
    A = oracle_mod.allowed_matrix(cu, m)
    cov, per_unit, empty = coverage(wl, T, T, hq, tile_m, tile_n)
    for h in range(hq):
        np.testing.assert_array_equal(cov[h], A.astype(np.int32))
    assert empty == 0
    np.testing.assert_array_equal(per_unit, wl["unit_pairs"])
    assert wl["pairs_per_head"] == int(A.sum())
    # cost = pairs + c_tile * (sub-tiles x kv tiles computed + sub-tiles)
    for u, c, p in zip(wl["units"], wl["unit_cost"], wl["unit_pairs"]):
        nsub = 2 if u[5] >= 0 else 1
        tiles = sum(int(wl["runs"][r][2] - wl["runs"][r][1]) for r in range(u[7], u[7] + u[8]))
        assert c == p + 3 * (nsub * tiles + nsub)


@pytest.mark.parametrize("cp", [2, 3])
def test_worklist_zigzag_pairs_cover_once(oracle_mod, cp):
    lengths = [19, 7, 2, 30, 0, 12]
    cu = W.cu_seqlens_of(lengths)
    for r in range(cp):
        tq = oracle_mod.zigzag_map(cu, cp, r)[0].shape[0]
        for s in range(cp):
            tk = oracle_mod.zigzag_map(cu, cp, s)[0].shape[0]
            m = oracle_mod.Mask(W.MASK_ZIGZAG_PAIR, cp=cp, q_rank=r, k_rank=s)
            wl = oracle_mod.worklist(cu, m, 4, 4, 2, 1, num_ctas=3)
            A = oracle_mod.allowed_matrix(cu, m, Tq=tq, Tk=tk)
            cov, per_unit, empty = coverage(wl, tq, tk, 2, 4, 4)
            for h in range(2):
                np.testing.assert_array_equal(cov[h], A.astype(np.int32))
            assert empty == 0
            np.testing.assert_array_equal(per_unit, wl["unit_pairs"])


def test_worklist_explicit_slices(oracle_mod):
    # two q segments; the second sees a FULL block and a shifted causal block
    sl = np.array([[0, 10, 0, 0, 10, 0, 1, 0],
                   [10, 9, 30, 0, 6, 0, 0, 0],
                   [10, 9, 30, 10, 12, 25, 1, 4]], dtype=np.int32)
    m = oracle_mod.Mask(W.MASK_SLICES, slices=sl)
    cu = W.cu_seqlens_of([22])
    wl = oracle_mod.worklist(cu, m, 4, 4, 2, 2, num_ctas=2)
    A = oracle_mod.allowed_matrix(cu, m, Tq=22, Tk=22)
    cov, per_unit, empty = coverage(wl, 22, 22, 2, 4, 4)
    np.testing.assert_array_equal(cov[0], A.astype(np.int32))
    assert empty == 0
    assert len(wl["segs"]) == 2


def test_square_tiles_causal_doc_closed_form(oracle_mod):
    b, n = 8, 9
    cu = W.cu_seqlens_of([b * n])
    wl = oracle_mod.worklist(cu, oracle_mod.Mask(), b, b, 2, 1, num_ctas=4)
    tiles = sum(int(r[2] - r[1]) for r in wl["runs"])
    assert tiles == n * (n + 1) // 2


def test_worklist_csr_is_lpt_in_enumeration_order(oracle_mod):
    w = W.tiny_pack()
    wl = oracle_mod.worklist(w.cu_seqlens, oracle_mod.Mask(), 128, 128, 4, 4, num_ctas=7, c_tile=100)
    off = wl["cta_off"]
    units = wl["units"]
    assert off[0] == 0 and off[-1] == len(units) and np.all(np.diff(off) >= 0)
    assert sorted(units[:, 0].tolist()) == list(range(len(units)))
    # LPT over the enumeration-order costs gives the same bins
    cost_by_uid = np.zeros(len(units), dtype=np.int64)
    cost_by_uid[units[:, 0]] = wl["unit_cost"]
    assign, _, loads = oracle_mod.lpt(cost_by_uid, 7)
    for b in range(7):
        seg = units[off[b]:off[b + 1]]
        assert np.all(seg[:, 9] == b)
        assert np.all(assign[seg[:, 0]] == b)
        # a bin runs its units in enumeration order
        assert np.all(np.diff(seg[:, 0]) > 0)
        c = wl["unit_cost"][off[b]:off[b + 1]]
        assert c.sum() == loads[b]


def test_zigzag_chunk_without_keys_keeps_empty_segment(oracle_mod):
    # rank 0's first chunk (positions [0, m)) sees nothing of rank 1's chunks
    cp = 2
    cu = W.cu_seqlens_of([16])
    m = oracle_mod.Mask(W.MASK_ZIGZAG_PAIR, cp=cp, q_rank=0, k_rank=1)
    wl = oracle_mod.worklist(cu, m, 4, 4, 2, 2, num_ctas=2)
    segs = wl["segs"]
    assert len(segs) == 2 and segs[0][4] == 0 and segs[1][4] == 2
    empty_units = [u for u in wl["units"] if u[1] == 0]
    assert all(u[8] == 0 for u in empty_units)


# ------------------------------------------------------ run-time dispatch order
def test_dispatch_order_worked_examples(oracle_mod):
    # classes floor(log2(max(c, 1))): 100, 70, 120 -> 6; 40 -> 5; 20, 30 -> 4; 10 -> 3; 5 -> 2
    costs = [100, 70, 120, 40, 20, 40, 30, 10, 5]
    # one CTA: class 6 has 145 below it (>= 2^7), class 5 has 65 (>= 2^6), class 4
    # only 15 (< 2^5): classes 6 and 5 in uid order, then 30, 20, 10, 5 by cost
    assert oracle_mod.dispatch_order(costs, 1).tolist() == [0, 1, 2, 3, 5, 6, 4, 7, 8]
    # two CTAs: 145 < 2 * 2^7 already at class 6, so the whole order is LPT
    assert oracle_mod.dispatch_order(costs, 2).tolist() == [2, 0, 1, 3, 5, 6, 4, 7, 8]
    # the lowest class always takes the LPT order (nothing below it)
    assert oracle_mod.dispatch_order([1, 3, 2, 0], 1).tolist() == [1, 2, 0, 3]


def test_dispatch_order_is_lpt_over_power_of_two_classes(oracle_mod):
    """On a real worklist the order is a permutation of the uids: a prefix whose
    cost classes never increase, uids ascending inside a class, then a suffix
    of the lowest classes sorted by (cost desc, uid asc); the class of each cost
    is checked by integer shifts (2^k <= c < 2^(k+1)), and the suffix starts
    where the work left below a class drops under 152 * 2^(k+1)."""
    w = W.long_tail_gqa(1)
    wl = oracle_mod.worklist(w.cu_seqlens, oracle_mod.Mask(), 128, 128, w.num_q_heads,
                             w.num_kv_heads, 152, 65536)
    uid = wl["units"][:, 0]
    cost = np.zeros(uid.shape[0], dtype=np.int64)
    cost[uid] = wl["unit_cost"]
    order = oracle_mod.dispatch_order(cost, 152)
    assert sorted(order.tolist()) == list(range(uid.shape[0]))
    c = np.maximum(cost[order], 1)
    k = np.zeros_like(c)
    for e in range(63):
        k[(c >> e) >= 1] = e
    assert np.all((np.left_shift(1, k) <= c) & (c < np.left_shift(1, k + 1)))
    assert np.all(np.diff(k) <= 0)
    # the LPT suffix: from the first unit after which the order is cost-sorted
    # and whose class fails the absorption test
    cls_work = {int(x): int(cost[order][k == x].sum()) for x in np.unique(k)}
    fails = [x for x in sorted(cls_work, reverse=True)
             if sum(v for y, v in cls_work.items() if y < x) < 152 * 2 ** (x + 1)]
    split = fails[0]
    head = k > split
    assert 0 < head.sum() < len(order)
    assert np.all(head[:head.sum()]) and not np.any(head[head.sum():])
    kh, oh = k[head], order[head]
    assert np.all(np.diff(oh)[np.diff(kh) == 0] > 0)
    ct, ot = cost[order][~head], order[~head]
    assert np.all((np.diff(ct) < 0) | ((np.diff(ct) == 0) & (np.diff(ot) > 0)))


def _list_schedule(costs, order, m):
    """Graham's list scheduling: units in `order`, each started on the machine
    that becomes free first (lowest id on ties); returns the makespan."""
    free = [0] * m
    for u in order:
        b = min(range(m), key=lambda i: (free[i], i))
        free[b] += int(costs[u])
    return max(free)


def test_dispatch_order_list_scheduling_within_graham_bound(oracle_mod):
    """The pages' LPT rule assigns each unit to the least loaded worker.  Run
    at run time, "least loaded" is the worker that frees up first, i.e. list
    scheduling in the dispatch order, with a unit's cost as its duration.  For
    any order Graham's bound holds: makespan <= (2 - 1/m) OPT, with OPT found
    here by brute force over all assignments; with the order fully sorted by
    cost (every class at or below the split) the LPT bound 4/3 - 1/(3m) holds
    too."""
    rng = np.random.default_rng(11)
    for trial in range(80):
        n = int(rng.integers(1, 9))
        m = int(rng.integers(1, 4))
        costs = rng.integers(0, 300, size=n)
        order = oracle_mod.dispatch_order(costs, m)
        assert sorted(order.tolist()) == list(range(n))
        span = _list_schedule(costs, order, m)
        opt = min(max(np.bincount(np.array(a), weights=costs, minlength=m))
                  for a in itertools.product(range(m), repeat=n))
        assert span >= opt
        assert span * m <= (2 * m - 1) * opt + 1e-9
        srt = sorted(range(n), key=lambda u: (-int(costs[u]), u))
        if order.tolist() == srt:
            assert span * 3 * m <= (4 * m - 1) * opt + 1e-9


# ------------------------------------------------------ short documents sharing tiles
def test_packed_groups_hand_worked(oracle_mod):
    """"03 · 长文负载均衡" §4.1: a block shorter than a tile is charged as a whole
    tile.  With tile 16: documents 2-4 (1, 9, 0 rows; 12 would overflow), 5-6
    (12 + 3; 16 is not short) and 8-11 (4 x 4 = 16 rows) share tiles; 0, 12
    (alone in their group), 1 and 7 (not shorter than a tile) keep their own."""
    lengths = [5, 17, 1, 9, 0, 12, 3, 16, 4, 4, 4, 4, 15]
    cu = W.cu_seqlens_of(lengths)
    wl = oracle_mod.worklist(cu, oracle_mod.Mask(), 16, 16, 1, 1, num_ctas=2, pack_docs=1)
    sl, sm = wl["slices"], wl["slice_masks"]
    got = [(int(r[0]), int(r[1]), int(r[6])) for r in sl]
    c = [int(x) for x in cu]
    assert got == [(c[0], 5, 1), (c[1], 17, 1), (c[2], 10, 4), (c[5], 15, 4), (c[7], 16, 1),
                   (c[8], 16, 4), (c[12], 15, 1)]
    assert [int(x) for x in sm[2]] == [0b11, 0, 0, 0]           # rows 0 and 1 start documents
    assert [int(x) for x in sm[3]] == [1 | (1 << 12), 0, 0, 0]
    assert [int(x) for x in sm[5]] == [1 | (1 << 4) | (1 << 8) | (1 << 12), 0, 0, 0]
    # a packed slice is one q tile against one kv tile
    assert len(wl["segs"]) == 7 and all(int(g[4]) == 1 for g in wl["segs"])


PACK_CASES = [
    ([5, 17, 1, 9, 0, 12, 3, 16, 4, 4, 4, 4, 15], W.MASK_CAUSAL, {}),
    ([3, 1, 2, 7, 30, 2, 2, 0, 6, 1], W.MASK_SLIDING_WINDOW, {"window": 3}),
    ([8, 8, 8, 8, 1, 1], W.MASK_CAUSAL, {}),
]


@pytest.mark.parametrize("lengths,kind,kw", PACK_CASES)
@pytest.mark.parametrize("hq,hkv", [(2, 2), (3, 1)])
@pytest.mark.parametrize("tile", [8, 16])
def test_packed_worklist_covers_allowed_pairs_once(oracle_mod, lengths, kind, kw, hq, hkv, tile):
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    m = oracle_mod.Mask(kind, **kw)
    wl = oracle_mod.worklist(cu, m, tile, tile, hq, hkv, num_ctas=3, c_tile=2, pack_docs=1)
    plain = oracle_mod.worklist(cu, m, tile, tile, hq, hkv, num_ctas=3, c_tile=2)
    A = oracle_mod.allowed_matrix(cu, m)
    cov, per_unit, empty = coverage(wl, T, T, hq, tile, tile)
    for h in range(hq):
        np.testing.assert_array_equal(cov[h], A.astype(np.int32))
    assert empty == 0
    np.testing.assert_array_equal(per_unit, wl["unit_pairs"])
    assert wl["pairs_per_head"] == plain["pairs_per_head"] == int(A.sum())
    assert (wl["slices"][:, 6] == 4).any()
    # fewer computed tiles and fewer units than one tile grid per document
    def tiles(w):
        return sum((2 if u[5] >= 0 else 1) * sum(int(w["runs"][r][2] - w["runs"][r][1])
                                                 for r in range(u[7], u[7] + u[8]))
                   for u in w["units"])
    assert tiles(wl) < tiles(plain) and len(wl["units"]) < len(plain["units"])
