"""Pins of the CPU oracle against what the pages and mathematics fix.

None of these tests calls the CUDA library.  Each one checks an oracle
function against something other than itself: a closed form, a value printed
on the pages (tests/golden/), a library routine on tiny inputs
(torch.nn.functional.scaled_dot_product_attention in float64), brute force,
or an invariant of the method.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from packed_varlen_attention_cu_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(x):
    import torch
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rand_qkv(tq, tk, hq, hkv, d, seed, scale=1.0):
    q, k, v = W.make_qkv(tq, tk, hq, hkv, d, seed, scale)
    return q, k, v


# --------------------------------------------------------------------------
# Pair counts: the work term of "03 · 长文负载均衡" §1.1 in closed form.
# --------------------------------------------------------------------------
def test_causal_pair_count_closed_form(oracle_mod):
    for lengths in (W.tiny_pack().lengths, [1, 2, 3, 0, 5], W.long_tail_gqa(2).lengths):
        cu = W.cu_seqlens_of(lengths)
        want = sum(l * (l + 1) // 2 for l in lengths)
        assert oracle_mod.pair_count(cu, oracle_mod.Mask()) == want


def test_causal_pair_count_bruteforce_tiny(oracle_mod):
    cu = W.cu_seqlens_of([3, 1, 4, 1, 5])
    m = oracle_mod.Mask()
    assert oracle_mod.pair_count(cu, m, brute=True) == oracle_mod.pair_count(cu, m) == 6 + 1 + 10 + 1 + 15


def test_libra_example_golden(oracle_mod):
    g = _golden("libra_pair.json")
    a = oracle_mod.pair_count(W.cu_seqlens_of(g["lengths_A"]), oracle_mod.Mask())
    b = oracle_mod.pair_count(W.cu_seqlens_of(g["lengths_B"]), oracle_mod.Mask())
    assert a == g["pairs_A"] and b == g["pairs_B"]
    assert a * g["pairs_ratio_den"] == b * g["pairs_ratio_num"]
    sa = sum(l * l for l in g["lengths_A"])
    sb = sum(l * l for l in g["lengths_B"])
    assert sa == g["sum_sq_ratio"] * sb
    # "about 10x": the causal-pair ratio is within 0.03% of 10
    assert abs(a / b - 10.0) < 3e-3


def test_structured_mask_pair_counts_golden(oracle_mod):
    g = _golden("structured_masks.json")
    sq = g["shared_question"]
    cu = W.cu_seqlens_of([sq["question"]] + sq["answers"])
    got = oracle_mod.pair_count(cu, oracle_mod.Mask(W.MASK_SHARED_QUESTION, num_prefix=1))
    Q = sq["question"]
    closed = Q * (Q + 1) // 2 + sum(a * Q + a * (a + 1) // 2 for a in sq["answers"])
    assert got == closed == sq["pairs_per_head"]
    sw = g["sliding_window"]
    w = sw["window"]
    cu = W.cu_seqlens_of(sw["lengths"])
    got = oracle_mod.pair_count(cu, oracle_mod.Mask(W.MASK_SLIDING_WINDOW, window=w))
    closed = sum(l * (l + 1) // 2 if l <= w else w * (w + 1) // 2 + (l - w) * w for l in sw["lengths"])
    assert got == closed == sw["pairs_per_head"]


def test_window_one_and_huge(oracle_mod):
    cu = W.cu_seqlens_of([7, 3, 9])
    assert oracle_mod.pair_count(cu, oracle_mod.Mask(W.MASK_SLIDING_WINDOW, window=1)) == 19
    assert (oracle_mod.pair_count(cu, oracle_mod.Mask(W.MASK_SLIDING_WINDOW, window=100))
            == oracle_mod.pair_count(cu, oracle_mod.Mask()))


# --------------------------------------------------------------------------
# Zigzag maps: "03 · 长文负载均衡" §4.2 (rank i owns chunks i and 2cp-1-i)
# and §4.3 (per-document sharding gives every worker equal work).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("cp", [1, 2, 3, 8])
def test_zigzag_single_doc_equal_work(oracle_mod, cp):
    m = 5
    ell = 2 * cp * m
    cu = W.cu_seqlens_of([ell])
    per_rank = []
    for r in range(cp):
        gmap, table = oracle_mod.zigzag_map(cu, cp, r)
        assert list(table[0, :, 1]) == [r, 2 * cp - 1 - r]
        # each rank's rows attend to every earlier token of the document: sum (pos + 1)
        per_rank.append(int(np.sum(gmap.astype(np.int64) + 1)))
    closed = m * m * (2 * cp - 1) + m * (m + 1)
    assert per_rank == [closed] * cp
    assert sum(per_rank) == ell * (ell + 1) // 2


def test_zigzag_pairs_sum_over_kv_ranks(oracle_mod):
    """Per-rank causal work summed over the ring equals the rank's own count."""
    cp = 4
    lengths = [37, 8, 1, 0, 64, 13]
    cu = W.cu_seqlens_of(lengths)
    total = 0
    for r in range(cp):
        gmap, _ = oracle_mod.zigzag_map(cu, cp, r)
        tq = gmap.shape[0]
        rank_pairs = 0
        for s in range(cp):
            tk = oracle_mod.zigzag_map(cu, cp, s)[0].shape[0]
            rank_pairs += oracle_mod.pair_count(
                cu, oracle_mod.Mask(W.MASK_ZIGZAG_PAIR, cp=cp, q_rank=r, k_rank=s), Tq=tq, Tk=tk)
        docs = np.searchsorted(cu, gmap, side="right") - 1
        assert rank_pairs == int(np.sum(gmap - cu[docs] + 1))
        total += rank_pairs
    assert total == sum(l * (l + 1) // 2 for l in lengths)


def test_zigzag_union_and_remainder_rule(oracle_mod):
    cp = 3
    lengths = [17, 6, 5, 0, 1, 12]
    cu = W.cu_seqlens_of(lengths)
    seen = []
    for r in range(cp):
        gmap, table = oracle_mod.zigzag_map(cu, cp, r)
        seen.append(gmap)
        for d, ell in enumerate(lengths):
            for e, c in enumerate((r, 2 * cp - 1 - r)):
                want_len = ell // (2 * cp) + (1 if c < ell % (2 * cp) else 0)
                assert table[d, e, 3] == want_len
                # chunks are contiguous in chunk order: offset = sum of earlier chunk lengths
                off = sum(ell // (2 * cp) + (1 if cc < ell % (2 * cp) else 0) for cc in range(c))
                assert table[d, e, 2] == cu[d] + off
    allr = np.sort(np.concatenate(seen))
    assert np.array_equal(allr, np.arange(cu[-1]))


def test_zigzag_ragged_doc_imbalance_small(oracle_mod):
    cp, ell = 8, 16005
    cu = W.cu_seqlens_of([ell])
    work = [int(np.sum(oracle_mod.zigzag_map(cu, cp, r)[0].astype(np.int64) + 1)) for r in range(cp)]
    assert sum(work) == ell * (ell + 1) // 2
    assert (max(work) - min(work)) / (sum(work) / cp) < 1e-3


# --------------------------------------------------------------------------
# Attention: textbook definitions and library routines on tiny inputs.
# --------------------------------------------------------------------------
def _mask_blocks(lengths):
    """Per-document causal mask built as a block diagonal of lower triangles."""
    import torch
    return torch.block_diag(*[torch.tril(torch.ones(l, l, dtype=torch.bool)) for l in lengths if l > 0])


def _sdpa(q, k, v, allowed, hq, hkv):
    """float64 SDPA on CPU with an explicit boolean mask; kv head of q head h is h // (hq/hkv)."""
    import torch
    G = hq // hkv
    qd = q.double().permute(1, 0, 2)          # [Hq, T, d]
    kd = k.double()[:, torch.arange(hq) // G].permute(1, 0, 2)
    vd = v.double()[:, torch.arange(hq) // G].permute(1, 0, 2)
    out = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, attn_mask=allowed)
    return out.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (3, 1), (6, 2)])
def test_attention_matches_sdpa_causal_docs(oracle_mod, hq, hkv):
    lengths = [5, 1, 9, 3, 14]
    cu = W.cu_seqlens_of(lengths)
    T = cu[-1]
    q, k, v = _rand_qkv(T, T, hq, hkv, 16, seed=3)
    out, lse = oracle_mod.attention(_bits(q), _bits(k), _bits(v), cu, oracle_mod.Mask())
    ref = _sdpa(q, k, v, _mask_blocks(lengths), hq, hkv)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_attention_matches_sdpa_window_and_shared_question(oracle_mod):
    import torch
    lengths = [11, 4, 13]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = _rand_qkv(T, T, 4, 2, 8, seed=5)
    w = 3
    band = torch.block_diag(*[torch.tril(torch.ones(l, l, dtype=torch.bool))
                              & ~torch.tril(torch.ones(l, l, dtype=torch.bool), diagonal=-w)
                              for l in lengths])
    out, _ = oracle_mod.attention(_bits(q), _bits(k), _bits(v), cu,
                                  oracle_mod.Mask(W.MASK_SLIDING_WINDOW, window=w))
    np.testing.assert_allclose(out, _sdpa(q, k, v, band, 4, 2), rtol=1e-10, atol=1e-12)
    # shared question: doc 0 is the question; answers see the question fully and themselves causally
    sq = _mask_blocks(lengths).clone()
    sq[cu[1]:, : cu[1]] = True
    out, _ = oracle_mod.attention(_bits(q), _bits(k), _bits(v), cu,
                                  oracle_mod.Mask(W.MASK_SHARED_QUESTION, num_prefix=1))
    np.testing.assert_allclose(out, _sdpa(q, k, v, sq, 4, 2), rtol=1e-10, atol=1e-12)


def test_attention_bruteforce_softmax_and_lse(oracle_mod):
    """Direct exp / sum without max subtraction, fp64, tiny pack."""
    lengths = [6, 2, 7]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    hq, hkv, d = 2, 1, 8
    q, k, v = _rand_qkv(T, T, hq, hkv, d, seed=11)
    out, lse = oracle_mod.attention(_bits(q), _bits(k), _bits(v), cu, oracle_mod.Mask(), scale=0.3)
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    for h in range(hq):
        for i in range(T):
            doc = np.searchsorted(cu, i, side="right") - 1
            js = np.arange(cu[doc], i + 1)
            e = np.exp(0.3 * (kd[js, 0] @ qd[i, h]))
            np.testing.assert_allclose(out[i, h], (e[:, None] * vd[js, 0]).sum(0) / e.sum(), rtol=1e-12)
            assert abs(lse[h, i] - math.log(e.sum())) < 1e-12


def test_attention_special_cases(oracle_mod):
    lengths = [9, 5]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = _rand_qkv(T, T, 2, 2, 8, seed=2)
    # window 1: every row sees only itself -> O_i = v_i and LSE_i = scale q_i.k_i
    out, lse = oracle_mod.attention(_bits(q), _bits(k), _bits(v), cu,
                                    oracle_mod.Mask(W.MASK_SLIDING_WINDOW, window=1))
    np.testing.assert_array_equal(out, v.double().numpy())
    s = (q.double() * k.double()).sum(-1).numpy() / math.sqrt(8)
    np.testing.assert_allclose(lse, s.T, rtol=1e-13)
    # constant V within each document -> O equals that constant
    vc = v.clone()
    for dd in range(len(lengths)):
        vc[cu[dd]:cu[dd + 1]] = v[cu[dd]]
    out, _ = oracle_mod.attention(_bits(q), _bits(k), _bits(vc), cu, oracle_mod.Mask())
    for dd in range(len(lengths)):
        np.testing.assert_allclose(out[cu[dd]:cu[dd + 1]],
                                   np.broadcast_to(vc[cu[dd]].double().numpy(),
                                                   (lengths[dd], 2, 8)), rtol=1e-12)


def test_single_doc_is_standard_causal(oracle_mod):
    import torch
    T, H, d = 33, 2, 16
    q, k, v = _rand_qkv(T, T, H, H, d, seed=7)
    out, _ = oracle_mod.attention(_bits(q), _bits(k), _bits(v), W.cu_seqlens_of([T]), oracle_mod.Mask())
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double().permute(1, 0, 2), k.double().permute(1, 0, 2), v.double().permute(1, 0, 2),
        is_causal=True).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_packed_equals_docs_alone(oracle_mod):
    lengths = [13, 4, 21]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = _rand_qkv(T, T, 2, 1, 8, seed=9)
    out, lse = oracle_mod.attention(_bits(q), _bits(k), _bits(v), cu, oracle_mod.Mask())
    for dd, l in enumerate(lengths):
        a, b = cu[dd], cu[dd + 1]
        o1, l1 = oracle_mod.attention(_bits(q[a:b]), _bits(k[a:b]), _bits(v[a:b]),
                                      W.cu_seqlens_of([l]), oracle_mod.Mask())
        np.testing.assert_allclose(out[a:b], o1, rtol=1e-12)
        np.testing.assert_allclose(lse[:, a:b], l1, rtol=1e-12)


def test_brute_candidates_agree(oracle_mod):
    lengths = [7, 0, 12, 5]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = _rand_qkv(T, T, 2, 2, 8, seed=4)
    for m in (oracle_mod.Mask(), oracle_mod.Mask(W.MASK_SLIDING_WINDOW, window=4),
              oracle_mod.Mask(W.MASK_SHARED_QUESTION, num_prefix=1)):
        a = oracle_mod.attention(_bits(q), _bits(k), _bits(v), cu, m)
        b = oracle_mod.attention(_bits(q), _bits(k), _bits(v), cu, m, brute=True)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


def test_sampled_jobs_equal_full(oracle_mod):
    lengths = [10, 17]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = _rand_qkv(T, T, 4, 2, 8, seed=8)
    full_o, full_l = oracle_mod.attention(_bits(q), _bits(k), _bits(v), cu, oracle_mod.Mask())
    jobs = W.random_rows(T, 4, 20, seed=1)
    o, l = oracle_mod.attention(_bits(q), _bits(k), _bits(v), cu, oracle_mod.Mask(), jobs=jobs)
    np.testing.assert_array_equal(o, full_o[jobs[:, 0], jobs[:, 1]])
    np.testing.assert_array_equal(l, full_l[jobs[:, 1], jobs[:, 0]])


# --------------------------------------------------------------------------
# Merge: "03 · 长文负载均衡" §3.2 (DCP online-softmax rescale-and-sum) and the
# ring-attention loop of "长序列训练与上下文并行": merging partials over any
# split of the keys equals attention over all keys.
# --------------------------------------------------------------------------
def test_merge_over_kv_split_equals_unsplit(oracle_mod):
    T, hq, hkv, d = 23, 2, 1, 8
    q, k, v = _rand_qkv(T, T, hq, hkv, d, seed=12)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    full = np.array([[0, T, 0, 0, T, 0, 1, 0]], dtype=np.int32)
    o, l = oracle_mod.attention(qb, kb, vb, W.cu_seqlens_of([T]), oracle_mod.Mask(W.MASK_SLICES, slices=full))
    for x in (1, 9, 22):
        a = np.array([[0, T, 0, 0, x, 0, 1, 0]], dtype=np.int32)
        b = np.array([[0, T, 0, x, T - x, x, 1, 0]], dtype=np.int32)
        oa, la = oracle_mod.attention(qb, kb, vb, W.cu_seqlens_of([T]), oracle_mod.Mask(W.MASK_SLICES, slices=a))
        ob, lb = oracle_mod.attention(qb, kb, vb, W.cu_seqlens_of([T]), oracle_mod.Mask(W.MASK_SLICES, slices=b))
        # rows before x see nothing of part b -> lse -inf there
        assert np.all(np.isneginf(lb[:, :x]))
        om, lm = oracle_mod.merge(oa, la, ob, lb)
        np.testing.assert_allclose(om, o, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lm, l, rtol=1e-12)
        om2, lm2 = oracle_mod.merge(ob, lb, oa, la)
        np.testing.assert_allclose(om2, om, rtol=1e-14)


def test_merge_neg_inf_identity(oracle_mod):
    rng = np.random.default_rng(0)
    oa = rng.standard_normal((5, 3, 4))
    la = rng.standard_normal((3, 5))
    ob = rng.standard_normal((5, 3, 4))
    lb = np.full((3, 5), -np.inf)
    o, l = oracle_mod.merge(oa, la, ob, lb)
    np.testing.assert_allclose(o, oa, rtol=1e-15)
    np.testing.assert_array_equal(l, la)
    o, l = oracle_mod.merge(np.zeros_like(oa), lb, ob * 0, lb)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_zigzag_ring_merge_equals_unsharded(oracle_mod):
    cp = 3
    lengths = [19, 7, 2, 30]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    hq, hkv, d = 2, 1, 8
    q, k, v = _rand_qkv(T, T, hq, hkv, d, seed=13)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    full_o, full_l = oracle_mod.attention(qb, kb, vb, cu, oracle_mod.Mask())
    maps = [oracle_mod.zigzag_map(cu, cp, r)[0] for r in range(cp)]
    for r in range(cp):
        acc_o = acc_l = None
        for t in range(cp):
            s = (r - t) % cp
            m = oracle_mod.Mask(W.MASK_ZIGZAG_PAIR, cp=cp, q_rank=r, k_rank=s)
            o, l = oracle_mod.attention(qb[maps[r]], kb[maps[s]], vb[maps[s]], cu, m)
            if acc_o is None:
                acc_o, acc_l = o, l
            else:
                acc_o, acc_l = oracle_mod.merge(acc_o, acc_l, o, l)
        np.testing.assert_allclose(acc_o, full_o[maps[r]], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(acc_l, full_l[:, maps[r]], rtol=1e-12)


# --------------------------------------------------------------------------
# LPT: "03 · 长文负载均衡" §2.1 and "数据并行负载均衡" §4.4 phase 1.
# --------------------------------------------------------------------------
def test_lpt_hand_worked_golden(oracle_mod):
    for ex in _golden("lpt_examples.json")["hand_worked"]:
        assign, order, loads = oracle_mod.lpt(ex["costs"], ex["bins"])
        assert list(assign) == ex["assign"]
        assert list(loads) == ex["loads"]


@pytest.mark.parametrize("m", [2, 3, 5, 8])
def test_lpt_graham_tight_instance(oracle_mod, m):
    costs = [c for j in range(2 * m - 1, m, -1) for c in (j, j)] + [m, m, m]
    _, _, loads = oracle_mod.lpt(costs, m)
    assert loads.max() == 4 * m - 1
    assert loads.sum() == sum(costs) == 3 * m * m


def test_lpt_vs_bruteforce_optimum(oracle_mod):
    rng = np.random.default_rng(5)
    for trial in range(60):
        n = int(rng.integers(1, 10))
        bins = int(rng.integers(1, 4))
        costs = rng.integers(1, 50, size=n)
        _, _, loads = oracle_mod.lpt(costs, bins)
        opt = min(max(np.bincount(np.array(a), weights=costs, minlength=bins))
                  for a in itertools.product(range(bins), repeat=n))
        assert loads.max() >= opt
        assert loads.max() * 3 * bins <= (4 * bins - 1) * opt + 1e-9
        assert loads.sum() == costs.sum()


def test_lpt_fewer_items_than_bins_and_determinism(oracle_mod):
    costs = [3, 8, 8, 1]
    a, o, _ = oracle_mod.lpt(costs, 10)
    assert list(o) == [1, 2, 0, 3] and list(a) == [2, 0, 1, 3]
    a2, o2, _ = oracle_mod.lpt(costs, 10)
    assert np.array_equal(a, a2) and np.array_equal(o, o2)
