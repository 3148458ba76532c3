"""Sharding solvers on the GPU against the oracle ("03 · 长文负载均衡" §4.2-§4.4):
chunk areas, min-heap dispatch and striped maps bit for bit, and a dispatched
pack run rank by rank (AttnSlices over the full K/V) equal to the unsharded
oracle."""
import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import api
from packed_varlen_attention_cu_gb300 import workloads as W

from gpu_util import compare, oracle_mask, run_gpu, to_np

pytestmark = pytest.mark.gpu

MASKS = [(W.MASK_CAUSAL, {}), (W.MASK_SLIDING_WINDOW, {"window": 300}),
         (W.MASK_SHARED_QUESTION, {"num_prefix_docs": 2})]


def _areas(cu_np, kind, kw, cs):
    T = int(cu_np[-1])
    cu = torch.from_numpy(cu_np).cuda()
    m = api.make_mask(kind, T, T, **kw)
    a = api.chunk_areas(cu, m, cs)
    torch.cuda.synchronize()
    return a.cpu().numpy()


@pytest.mark.parametrize("kind,kw", MASKS)
def test_chunk_areas_bit_exact(oracle_mod, kind, kw):
    okw = {"window": kw.get("window", 0), "num_prefix": kw.get("num_prefix_docs", 0)}
    for cu_np, cs in ((W.tiny_pack().cu_seqlens, 100), (W.tiny_pack().cu_seqlens, 1),
                      (W.cu_seqlens_of([5000, 3, 20000, 777]), 1024)):
        got = _areas(cu_np, kind, kw, cs)
        want = oracle_mod.chunk_areas(cu_np, oracle_mask(kind, **okw), cs)
        np.testing.assert_array_equal(got, want)


def test_chunk_areas_128k_pack(oracle_mod):
    w = W.zigzag_pack()
    got = _areas(w.cu_seqlens, W.MASK_CAUSAL, {}, 1024)
    np.testing.assert_array_equal(got, oracle_mod.chunk_areas(w.cu_seqlens, oracle_mask(W.MASK_CAUSAL), 1024))
    assert int(got.sum()) == 488185982


def _dispatch(areas, cp):
    a = torch.from_numpy(np.ascontiguousarray(areas, dtype=np.int64)).cuda()
    b, l = api.dispatch_chunks(a, cp)
    torch.cuda.synchronize()
    return b.cpu().numpy(), l.cpu().numpy()


@pytest.mark.parametrize("case", ["128k", "random_max", "ties", "one_each", "zeros"])
def test_dispatch_bit_exact(oracle_mod, case):
    rng = np.random.default_rng(3)
    if case == "128k":
        w = W.zigzag_pack()
        areas, cp = oracle_mod.chunk_areas(w.cu_seqlens, oracle_mask(W.MASK_CAUSAL), 1024), 8
    elif case == "random_max":
        areas, cp = rng.integers(0, 1 << 40, size=8192), 1024
    elif case == "ties":
        areas, cp = rng.integers(0, 4, size=960), 24
    elif case == "one_each":
        areas, cp = rng.integers(0, 100, size=64), 64
    else:
        areas, cp = np.zeros(32, dtype=np.int64), 4
    got_b, got_l = _dispatch(areas, cp)
    want_b, want_l = oracle_mod.dispatch_minheap(areas, cp)
    np.testing.assert_array_equal(got_b, want_b)
    np.testing.assert_array_equal(got_l, want_l)


@pytest.mark.parametrize("T,cp,stripe", [(131072, 8, 1), (131072, 8, 1024), (1000, 3, 7), (5, 8, 2)])
def test_striped_bit_exact(oracle_mod, T, cp, stripe):
    for r in range(cp):
        n = api.striped_shard_len(T, cp, r, stripe)
        m = torch.full((max(n, 1),), -1, dtype=torch.int32, device="cuda")
        api.striped_shard(T, cp, r, stripe, m)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(m.cpu().numpy()[:n], oracle_mod.striped_map(T, cp, r, stripe))


def _rank_slices(cu, chunks, cs, T):
    """AttnSlices of one rank: its chunks, in chunk order, as rank-local query rows
    against the full pack's keys (causal within each document)."""
    rows, sl = [], []
    local = 0
    for c in sorted(chunks):
        a, b = c * cs, min((c + 1) * cs, T)
        rows.append(np.arange(a, b, dtype=np.int32))
        for d in range(len(cu) - 1):
            lo, hi = max(a, cu[d]), min(b, cu[d + 1])
            if lo < hi:
                sl.append([local + lo - a, hi - lo, lo - cu[d], cu[d], cu[d + 1] - cu[d], 0, 1, 0])
        local += b - a
    return np.concatenate(rows), np.array(sl, dtype=np.int32)


def test_dispatched_pack_equals_unsharded(oracle_mod):
    lengths = [900, 5, 300, 1300, 64, 1, 430]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    hq, hkv, d, cp, cs = 4, 2, 128, 4, 125
    n = (T + cs - 1) // cs
    assert n % cp == 0
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 17)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    areas = api.chunk_areas(torch.from_numpy(cu).cuda(), api.make_mask(W.MASK_CAUSAL, T, T), cs)
    bucket, loads = api.dispatch_chunks(areas, cp)
    torch.cuda.synchronize()
    bucket = bucket.cpu().numpy()
    o_full = np.zeros((T, hq, d))
    l_full = np.zeros((hq, T))
    for r in range(cp):
        rows, sl = _rank_slices(cu, np.nonzero(bucket == r)[0], cs, T)
        qr = qd[torch.from_numpy(rows).long().cuda()].contiguous()
        m = api.make_mask(W.MASK_SLICES, rows.shape[0], T, slices=sl)
        o, l, _ = run_gpu(qr, kd, vd, cu, m, hq, hkv, out_fp32=True)
        o_full[rows] = to_np(o)
        l_full[:, rows] = to_np(l)
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu, oracle_mask(W.MASK_CAUSAL))
    compare(o_full, l_full, ref_o, ref_l, "dispatched pack")
    # the buckets' areas add up to the pack's pairs and are balanced by the greedy
    assert int(loads.sum().item()) == oracle_mod.pair_count(cu, oracle_mask(W.MASK_CAUSAL))
