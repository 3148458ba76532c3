"""Pins of the oracle's zigzag ring-step mask (every rank's step t at once).

"长序列训练与上下文并行", ring attention: cp ranks each hold a shard of Q and
of K/V; at step t rank r computes its Q against the K/V that started on rank
(r - t) mod cp, and the partial results of the cp steps are merged by online
softmax.  "03 · 长文负载均衡" §4.2-4.3: each rank's shard is the zigzag pair of
chunks (r, 2cp-1-r) of every document.  Rows are in ring order: rank 0's shard,
then rank 1's, and so on.

What the definitions fix, checked here without the oracle's own derivation:
- over the cp steps, every allowed pair of the causal per-document mask is
  met exactly once (the ring visits every K/V shard once), written out as a
  numpy block-diagonal triangle;
- the block of step t between the rows of rank r and of rank (r - t) mod cp
  is exactly the zigzag-pair mask of those ranks, and every other block is
  empty;
- per-step attention merged over the steps equals unsharded attention;
- the worklist of a step covers each of its allowed pairs exactly once.
"""
import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import workloads as W

from test_oracle_worklist import coverage

LENGTHS = [19, 7, 2, 30, 0, 12, 1, 45]


def _causal_docs(cu):
    """Causal per-document mask by definition (block-diagonal lower triangles)."""
    T = int(cu[-1])
    A = np.zeros((T, T), dtype=bool)
    for a, b in zip(cu[:-1], cu[1:]):
        n = int(b - a)
        A[a:b, a:b] = np.tril(np.ones((n, n), dtype=bool))
    return A


def _ring_order(oracle_mod, cu, cp):
    maps = [oracle_mod.zigzag_map(cu, cp, r)[0] for r in range(cp)]
    return np.concatenate(maps), np.cumsum([0] + [len(m) for m in maps])


@pytest.mark.parametrize("cp", [1, 2, 3, 4])
def test_ring_steps_partition_the_causal_mask(oracle_mod, cp):
    cu = W.cu_seqlens_of(LENGTHS)
    T = int(cu[-1])
    perm, _ = _ring_order(oracle_mod, cu, cp)
    assert np.array_equal(np.sort(perm), np.arange(T))
    np.testing.assert_array_equal(oracle_mod.ring_map(cu, cp), perm)
    hits = np.zeros((T, T), dtype=np.int32)
    for t in range(cp):
        A = oracle_mod.allowed_matrix(cu, oracle_mod.Mask(W.MASK_ZIGZAG_STEP, cp=cp, ring_step=t))
        hits[np.ix_(perm, perm)] += A.astype(np.int32)
    np.testing.assert_array_equal(hits, _causal_docs(cu).astype(np.int32))


@pytest.mark.parametrize("cp", [2, 3])
def test_ring_step_blocks_are_the_pair_masks(oracle_mod, cp):
    cu = W.cu_seqlens_of(LENGTHS)
    _, off = _ring_order(oracle_mod, cu, cp)
    for t in range(cp):
        A = oracle_mod.allowed_matrix(cu, oracle_mod.Mask(W.MASK_ZIGZAG_STEP, cp=cp, ring_step=t))
        for r in range(cp):
            for s in range(cp):
                blk = A[off[r]:off[r + 1], off[s]:off[s + 1]]
                if s == (r - t) % cp:
                    P = oracle_mod.allowed_matrix(
                        cu, oracle_mod.Mask(W.MASK_ZIGZAG_PAIR, cp=cp, q_rank=r, k_rank=s),
                        Tq=off[r + 1] - off[r], Tk=off[s + 1] - off[s])
                    np.testing.assert_array_equal(blk, P)
                else:
                    assert not blk.any()


def test_ring_step_attention_merged_equals_unsharded(oracle_mod):
    cp = 3
    cu = W.cu_seqlens_of(LENGTHS)
    T = int(cu[-1])
    hq, hkv, d = 4, 2, 16
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 21)
    perm, _ = _ring_order(oracle_mod, cu, cp)
    pt = torch.from_numpy(perm).long()
    qb, kb, vb = (oracle_mod.bf16_bits(x[pt]) for x in (q, k, v))
    acc_o = acc_l = None
    for t in range(cp):
        o, l = oracle_mod.attention(qb, kb, vb, cu,
                                    oracle_mod.Mask(W.MASK_ZIGZAG_STEP, cp=cp, ring_step=t))
        if acc_o is None:
            acc_o, acc_l = o, l
        else:
            acc_o, acc_l = oracle_mod.merge(acc_o, acc_l, o, l)
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu, oracle_mod.Mask())
    np.testing.assert_allclose(acc_o, ref_o[perm], atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(acc_l, ref_l[:, perm], atol=1e-12, rtol=1e-12)


@pytest.mark.parametrize("cp", [2, 3])
@pytest.mark.parametrize("hq,hkv", [(2, 1), (3, 1)])
def test_ring_step_worklist_covers_allowed_pairs_once(oracle_mod, cp, hq, hkv):
    cu = W.cu_seqlens_of(LENGTHS)
    T = int(cu[-1])
    for t in range(cp):
        m = oracle_mod.Mask(W.MASK_ZIGZAG_STEP, cp=cp, ring_step=t)
        wl = oracle_mod.worklist(cu, m, 4, 4, hq, hkv, num_ctas=3, c_tile=2)
        A = oracle_mod.allowed_matrix(cu, m)
        cov, per_unit, empty = coverage(wl, T, T, hq, 4, 4)
        for h in range(hq):
            np.testing.assert_array_equal(cov[h], A.astype(np.int32))
        assert empty == 0
        np.testing.assert_array_equal(per_unit, wl["unit_pairs"])
        assert wl["pairs_per_head"] == int(A.sum())
