"""Pins for the oracle's AttnSlice MaskTypes ("03 · 长文负载均衡" §4.4 names FULL,
CAUSAL, INV-CAUSAL and BI-CAUSAL; the geometry is the reading on token positions
stated in include/pva.h): the allowed matrix against the definitions written out
as loops, INV-CAUSAL attention as CAUSAL attention on the reversed sequence, the
BI-CAUSAL band, and the worklist's pair counts against the allowed matrix."""
import numpy as np
import pytest

import oracle
from packed_varlen_attention_cu_gb300 import workloads as W

FULL, CAUSAL, INV, BI = (oracle.SLICE_FULL, oracle.SLICE_CAUSAL, oracle.SLICE_INV_CAUSAL,
                         oracle.SLICE_BI_CAUSAL)


def _bits(x):
    return oracle.bf16_bits(x)


def _allowed_loops(slices, Tq, Tk):
    """The definitions, one pair at a time."""
    A = np.zeros((Tq, Tk), dtype=bool)
    for q_row0, q_len, q_pos0, k_row0, k_len, k_pos0, typ, w in slices:
        for i in range(q_row0, q_row0 + q_len):
            for j in range(k_row0, k_row0 + k_len):
                qp, kp = q_pos0 + (i - q_row0), k_pos0 + (j - k_row0)
                if typ == FULL:
                    ok = True
                elif typ == CAUSAL:
                    ok = kp <= qp and (w <= 0 or qp - kp < w)
                elif typ == INV:
                    ok = kp >= qp and (w <= 0 or kp - qp < w)
                else:
                    ok = kp >= qp and (k_pos0 + k_len) - kp >= (q_pos0 + q_len) - qp
                A[i, j] |= ok
    return A


CASES = [
    # square, start-aligned
    [[0, 12, 0, 0, 12, 0, INV, 0]],
    [[0, 12, 0, 0, 12, 0, INV, 4]],
    [[0, 12, 0, 0, 12, 0, BI, 0]],
    # rectangles and offset positions
    [[0, 7, 3, 0, 15, 3, BI, 0]],
    [[0, 7, 10, 2, 11, 5, INV, 0]],
    [[0, 9, 0, 0, 13, 2, BI, 0]],
    # mixed types over two query segments
    [[0, 10, 0, 0, 10, 0, CAUSAL, 3], [0, 10, 0, 10, 6, 0, INV, 0],
     [10, 5, 20, 4, 8, 18, BI, 0], [10, 5, 20, 12, 4, 30, FULL, 0]],
]


@pytest.mark.parametrize("slices", CASES)
def test_allowed_matrix_matches_definitions(slices):
    sl = np.array(slices, dtype=np.int32)
    Tq = int(max(s[0] + s[1] for s in slices))
    Tk = int(max(s[3] + s[4] for s in slices))
    A = oracle.allowed_matrix(W.cu_seqlens_of([Tq]), oracle.Mask(oracle.MASK_SLICES, slices=sl),
                              Tq, Tk)
    np.testing.assert_array_equal(A, _allowed_loops(slices, Tq, Tk))


def test_inv_causal_square_is_transposed_causal():
    L = 17
    c = np.array([[0, L, 0, 0, L, 0, CAUSAL, 0]], dtype=np.int32)
    i = np.array([[0, L, 0, 0, L, 0, INV, 0]], dtype=np.int32)
    cu = W.cu_seqlens_of([L])
    Ac = oracle.allowed_matrix(cu, oracle.Mask(oracle.MASK_SLICES, slices=c))
    Ai = oracle.allowed_matrix(cu, oracle.Mask(oracle.MASK_SLICES, slices=i))
    np.testing.assert_array_equal(Ai, Ac.T)


def test_bi_causal_band():
    # start-aligned q range of 5 against 9 keys: q <= k <= q + 4; square: the diagonal
    sl = np.array([[0, 5, 0, 0, 9, 0, BI, 0]], dtype=np.int32)
    A = oracle.allowed_matrix(W.cu_seqlens_of([5]), oracle.Mask(oracle.MASK_SLICES, slices=sl), 5, 9)
    for q in range(5):
        assert A[q].nonzero()[0].tolist() == list(range(q, q + 5))
    sq = np.array([[0, 6, 0, 0, 6, 0, BI, 0]], dtype=np.int32)
    A = oracle.allowed_matrix(W.cu_seqlens_of([6]), oracle.Mask(oracle.MASK_SLICES, slices=sq))
    np.testing.assert_array_equal(A, np.eye(6, dtype=bool))


def test_inv_causal_attention_is_reversed_causal_attention():
    # k >= q on positions 0..L-1 is k' <= q' on the reversed positions L-1-x
    L, hq, hkv, d = 19, 2, 1, 8
    q, k, v = W.make_qkv(L, L, hq, hkv, d, 31)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    inv = np.array([[0, L, 0, 0, L, 0, INV, 0]], dtype=np.int32)
    cau = np.array([[0, L, 0, 0, L, 0, CAUSAL, 0]], dtype=np.int32)
    cu = W.cu_seqlens_of([L])
    oi, li = oracle.attention(qb, kb, vb, cu, oracle.Mask(oracle.MASK_SLICES, slices=inv))
    oc, lc = oracle.attention(qb[::-1].copy(), kb[::-1].copy(), vb[::-1].copy(), cu,
                              oracle.Mask(oracle.MASK_SLICES, slices=cau))
    np.testing.assert_allclose(oi, oc[::-1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(li, lc[:, ::-1], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("slices", CASES[3:])
def test_worklist_pairs_match_allowed_matrix(slices):
    sl = np.array(slices, dtype=np.int32)
    Tq = int(max(s[0] + s[1] for s in slices))
    Tk = int(max(s[3] + s[4] for s in slices))
    m = oracle.Mask(oracle.MASK_SLICES, slices=sl)
    cu = W.cu_seqlens_of([Tq])
    A = oracle.allowed_matrix(cu, m, Tq, Tk)
    for tile in (4, 8):
        wl = oracle.worklist(cu, m, tile, tile, 2, 1, num_ctas=3)
        assert wl["pairs_per_head"] == int(A.sum())
