"""Pins for the oracle's attention backward: the analytic gradients match
central finite differences of a plain fp64 forward (itself checked against the
oracle forward), sum to zero over the keys where every row has a key, add up
over the q heads of a GQA group, and vanish for keys no query may see."""
import numpy as np
import pytest

import oracle
from packed_varlen_attention_cu_gb300 import workloads as W


def _bf16_values(x):
    """fp64 values of the bf16 bit patterns of x."""
    b = oracle.bf16_bits(x).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _forward(q, k, v, allowed, scale):
    """Masked softmax(scale Q K^T) V per head, GQA by contiguous groups, fp64."""
    Tq, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.zeros_like(q)
    for h in range(Hq):
        s = scale * q[:, h, :] @ k[:, h // G, :].T
        s = np.where(allowed, s, -np.inf)
        rows = allowed.any(1)
        m = np.where(rows, s.max(1), 0.0)
        p = np.where(allowed, np.exp(s - m[:, None]), 0.0)
        l = p.sum(1)
        out[rows, h, :] = (p[rows] / l[rows, None]) @ v[:, h // G, :]
    return out


@pytest.fixture(scope="module")
def case():
    cu = W.cu_seqlens_of([20, 7, 13])
    T, Hq, Hkv, d = 40, 4, 2, 8
    q, k, v = W.make_qkv(T, T, Hq, Hkv, d, 3)
    do = W.make_qkv(T, T, Hq, Hkv, d, 4)[0]
    return cu, q, k, v, do


def test_plain_forward_matches_oracle_forward(case):
    cu, q, k, v, do = case
    A = oracle.allowed_matrix(cu, oracle.Mask())
    scale = 1.0 / np.sqrt(q.shape[-1])
    ref, _ = oracle.attention(oracle.bf16_bits(q), oracle.bf16_bits(k), oracle.bf16_bits(v), cu,
                              oracle.Mask())
    got = _forward(_bf16_values(q), _bf16_values(k), _bf16_values(v), A, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_gradients_match_finite_differences(case):
    cu, q, k, v, do = case
    A = oracle.allowed_matrix(cu, oracle.Mask())
    scale = 1.0 / np.sqrt(q.shape[-1])
    qv, kv, vv, gv = (_bf16_values(x) for x in (q, k, v, do))
    dq, dk, dv = oracle.attention_bwd(oracle.bf16_bits(q), oracle.bf16_bits(k),
                                      oracle.bf16_bits(v), oracle.bf16_bits(do), cu, oracle.Mask())

    def loss(qq, kk, vv_):
        return float((gv * _forward(qq, kk, vv_, A, scale)).sum())

    rng = np.random.default_rng(0)
    eps = 1e-6
    for name, x, grad in (("q", qv, dq), ("k", kv, dk), ("v", vv, dv)):
        for _ in range(25):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, kv, vv), "k": (qv, xp, vv), "v": (qv, kv, xp)}[name]
            args_m = {"q": (xm, kv, vv), "k": (qv, xm, vv), "v": (qv, kv, xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_key_gradients_sum_to_zero(case):
    # sum_j dS_ij = 0 for every row with a key, so sum_j dK_j = 0 per kv head
    cu, q, k, v, do = case
    _, dk, _ = oracle.attention_bwd(oracle.bf16_bits(q), oracle.bf16_bits(k), oracle.bf16_bits(v),
                                    oracle.bf16_bits(do), cu, oracle.Mask())
    assert np.abs(dk.sum(0)).max() < 1e-12


def test_gqa_group_sums_per_head_gradients(case):
    cu, q, k, v, do = case
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    qb, kb, vb, gb = (oracle.bf16_bits(x) for x in (q, k, v, do))
    dq, dk, dv = oracle.attention_bwd(qb, kb, vb, gb, cu, oracle.Mask())
    # the same problem with every kv head repeated once per q head (MHA)
    kr, vr = np.repeat(kb, G, axis=1), np.repeat(vb, G, axis=1)
    dq2, dk2, dv2 = oracle.attention_bwd(qb, kr, vr, gb, cu, oracle.Mask())
    np.testing.assert_allclose(dq2, dq, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk2.reshape(dk2.shape[0], Hkv, G, -1).sum(2), dk, rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(dv2.reshape(dv2.shape[0], Hkv, G, -1).sum(2), dv, rtol=1e-12,
                               atol=1e-12)


def test_unseen_keys_get_no_gradient():
    # one slice: queries [0, 16) see keys [0, 10) causally; keys [10, 24) are never seen
    sl = np.array([[0, 16, 0, 0, 10, 0, oracle.SLICE_CAUSAL, 0]], dtype=np.int32)
    m = oracle.Mask(oracle.MASK_SLICES, slices=sl)
    q, _, _ = W.make_qkv(16, 16, 2, 2, 8, 9)
    _, k, v = W.make_qkv(24, 24, 2, 2, 8, 10)
    do = W.make_qkv(16, 16, 2, 2, 8, 11)[0]
    cu = W.cu_seqlens_of([16])
    dq, dk, dv = oracle.attention_bwd(oracle.bf16_bits(q), oracle.bf16_bits(k), oracle.bf16_bits(v),
                                      oracle.bf16_bits(do), cu, m)
    assert np.all(dk[10:] == 0) and np.all(dv[10:] == 0)
    assert np.abs(dk[:10]).max() > 0 and np.abs(dq).max() > 0


def test_sampled_jobs_equal_full_backward(case):
    # every sampled output equals the full backward's entry (both by definition)
    cu, q, k, v, do = case
    bits = [oracle.bf16_bits(x) for x in (q, k, v, do)]
    dq, dk, dv = oracle.attention_bwd(*bits, cu, oracle.Mask())
    qj = np.array([[0, 0], [7, 3], [19, 1], [20, 2], [39, 3], [27, 0]])
    kj = np.array([[0, 0], [5, 1], [19, 0], [26, 1], [39, 1]])
    sq, sk, sv = oracle.attention_bwd_jobs(*bits, cu, oracle.Mask(), qj, kj)
    np.testing.assert_allclose(sq, dq[qj[:, 0], qj[:, 1]], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(sk, dk[kj[:, 0], kj[:, 1]], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(sv, dv[kj[:, 0], kj[:, 1]], rtol=1e-12, atol=1e-13)
