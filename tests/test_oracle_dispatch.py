"""Pins for the oracle's dispatch and sharding solvers ("03 · 长文负载均衡"
§4.2-§4.4): chunk mask areas, MagiAttention's greedy min-heap dispatch,
striped maps and WLB-LLM's per-sequence / per-document choice.  Each is
checked against something other than itself: the pair count, the allowed
matrix, hand-worked examples, exhaustive search and closed forms."""
import itertools

import numpy as np
import pytest

import oracle
from packed_varlen_attention_cu_gb300 import workloads as W


@pytest.fixture(scope="module")
def o():
    return oracle


# ------------------------------------------------------------ chunk areas
@pytest.mark.parametrize("kind,kw", [(oracle.MASK_CAUSAL, {}),
                                     (oracle.MASK_SLIDING_WINDOW, {"window": 77}),
                                     (oracle.MASK_SHARED_QUESTION, {"num_prefix": 2})])
def test_chunk_areas_sum_to_pair_count(o, kind, kw):
    cu = W.cu_seqlens_of([300, 50, 1000, 7, 260])
    m = o.Mask(kind, **kw)
    a = o.chunk_areas(cu, m, 128)
    assert a.shape[0] == (int(cu[-1]) + 127) // 128
    assert int(a.sum()) == o.pair_count(cu, m)


def test_chunk_areas_brute_force(o):
    cu = W.cu_seqlens_of([37, 5, 60, 1, 21])
    T = int(cu[-1])
    for m in (o.Mask(), o.Mask(o.MASK_SLIDING_WINDOW, window=9),
              o.Mask(o.MASK_SHARED_QUESTION, num_prefix=1)):
        A = o.allowed_matrix(cu, m)
        for cs in (1, 7, 16, T + 3):
            a = o.chunk_areas(cu, m, cs)
            want = [int(A[c * cs:(c + 1) * cs].sum()) for c in range((T + cs - 1) // cs)]
            assert a.tolist() == want


def test_chunk_areas_rejects_rank_local_masks(o):
    cu = W.cu_seqlens_of([64])
    with pytest.raises(ValueError):
        o.chunk_areas(cu, o.Mask(o.MASK_ZIGZAG_PAIR, cp=2, q_rank=0, k_rank=0), 8)


# ------------------------------------------------------- min-heap dispatch
def test_dispatch_hand_worked_example(o):
    # areas 9..4, two buckets of 3: 9->B0, 8->B1, 7->B1 (8 < 9), 6->B0, 5->B0 (tie 15/15,
    # lower id), B0 full, 4->B1
    b, loads = o.dispatch_minheap([9, 8, 7, 6, 5, 4], 2)
    assert b.tolist() == [0, 1, 1, 0, 0, 1]
    assert loads.tolist() == [20, 19]


@pytest.mark.parametrize("cp", [2, 4, 8])
def test_dispatch_single_causal_doc_is_zigzag(o, cp):
    # One causal document cut into 2 cp equal chunks: chunk c pairs with 2 cp - 1 - c and
    # every bucket gets exactly the same area (the zigzag point of §4.2 / §4.4)
    m = 32
    cu = W.cu_seqlens_of([2 * cp * m])
    a = o.chunk_areas(cu, o.Mask(), m)
    b, loads = o.dispatch_minheap(a, cp)
    for c in range(cp):
        assert b[c] == b[2 * cp - 1 - c]
    assert len(set(loads.tolist())) == 1 and int(loads.sum()) == int(a.sum())


def _optimum(areas, cp):
    """Exhaustive minimum of the largest bucket over balanced assignments."""
    n = len(areas)
    cap = n // cp
    best = None

    def rec(i, fill, load):
        nonlocal best
        if i == n:
            v = max(load)
            best = v if best is None else min(best, v)
            return
        seen = set()
        for j in range(cp):
            if fill[j] == cap or (fill[j], load[j]) in seen:
                continue
            seen.add((fill[j], load[j]))
            fill[j] += 1
            load[j] += areas[i]
            rec(i + 1, fill, load)
            fill[j] -= 1
            load[j] -= areas[i]

    rec(0, [0] * cp, [0] * cp)
    return best


def test_dispatch_valid_and_near_optimal(o):
    rng = np.random.default_rng(5)
    worst = 0.0
    for trial in range(40):
        cp = int(rng.choice([2, 3, 4]))
        n = cp * int(rng.integers(1, 4))
        areas = rng.integers(0, 100, size=n).tolist()
        b, loads = o.dispatch_minheap(areas, cp)
        assert np.bincount(b, minlength=cp).tolist() == [n // cp] * cp
        assert [sum(a for a, x in zip(areas, b) if x == j) for j in range(cp)] == loads.tolist()
        opt = _optimum(areas, cp)
        assert max(loads) >= opt
        if opt:
            worst = max(worst, max(loads) / opt)
    assert worst < 1.5  # a greedy, not an exact solver (§4.4): close, not always optimal


def test_dispatch_needs_whole_buckets(o):
    with pytest.raises(ValueError):
        o.dispatch_minheap([1, 2, 3], 2)


# --------------------------------------------------------------- striped
@pytest.mark.parametrize("T,cp,stripe", [(100, 4, 1), (100, 4, 8), (7, 8, 2), (0, 2, 1)])
def test_striped_partition(o, T, cp, stripe):
    maps = [o.striped_map(T, cp, r, stripe) for r in range(cp)]
    allt = np.sort(np.concatenate(maps)) if T else np.zeros(0)
    assert allt.tolist() == list(range(T))
    for r, m in enumerate(maps):
        assert np.all(np.diff(m) > 0) and np.all((m // stripe) % cp == r)


def test_striped_causal_work_closed_form(o):
    # one causal document, stripe 1: rank r holds tokens r + k cp, k < K, whose causal
    # pairs sum to K (r + 1) + cp K (K - 1) / 2
    T, cp = 4096, 8
    K = T // cp
    for r in range(cp):
        m = o.striped_map(T, cp, r, 1)
        assert int((m + 1).sum()) == K * (r + 1) + cp * K * (K - 1) // 2


# ------------------------------------------------------------ WLB choice
def _brute_piece_tiles(p0, p1, tile):
    """(q tile, kv tile) pairs with an allowed causal pair, q tiles aligned at p0."""
    tiles = 0
    for r0 in range(p0, p1, tile):
        rows = np.arange(r0, min(r0 + tile, p1))
        for k0 in range(0, p1, tile):
            keys = np.arange(k0, k0 + tile)
            if (keys[None, :] <= rows[:, None]).any():
                tiles += 1
    return tiles


def _zz(len_, cp, c):
    base, rem = divmod(len_, 2 * cp)
    return c * base + min(c, rem), base + (1 if c < rem else 0)


def test_wlb_costs_brute_force(o):
    lengths = [70, 5, 300, 129, 1, 200]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    cp, tile, d = 2, 32, 64
    choice, costs = o.wlb_choose(cu, cp, tile, d)
    unit = tile * tile * 4 * d
    for r in range(cp):
        seq = doc = 0
        for c in (r, 2 * cp - 1 - r):
            off, ln = _zz(T, cp, c)
            for dd in range(len(lengths)):
                a, b = max(off, cu[dd]), min(off + ln, cu[dd + 1])
                if a < b:
                    seq += _brute_piece_tiles(a - cu[dd], b - cu[dd], tile)
            for dd in range(len(lengths)):
                off2, ln2 = _zz(lengths[dd], cp, c)
                if ln2:
                    doc += _brute_piece_tiles(off2, off2 + ln2, tile)
        assert costs[0, r] == seq * unit and costs[1, r] == doc * unit
    assert choice == (1 if costs[1].max() < costs[0].max() else 0)


def test_wlb_single_document_ties_to_per_sequence(o):
    cu = W.cu_seqlens_of([8192])
    choice, costs = o.wlb_choose(cu, 4, 128, 128)
    assert np.array_equal(costs[0], costs[1]) and choice == 0


def test_wlb_many_short_documents_prefer_per_sequence(o):
    # 64-token documents cut 2 cp = 8 ways: 8-token chunks, each charged a whole tile
    cu = W.cu_seqlens_of([64] * 64)
    choice, costs = o.wlb_choose(cu, 4, 128, 128)
    assert choice == 0 and costs[1].max() > 2 * costs[0].max()


def test_wlb_long_document_after_short_ones_prefers_per_document(o):
    # whole-pack zigzag puts the heavy end of the long document on the rank that also
    # holds the first chunk: per-document sharding balances it
    cu = W.cu_seqlens_of([256] * 16 + [16384])
    choice, costs = o.wlb_choose(cu, 4, 128, 128)
    assert choice == 1 and costs[1].max() < costs[0].max()
