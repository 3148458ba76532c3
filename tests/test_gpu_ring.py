"""Zigzag context parallelism on one GPU at cp = 8, against unsharded attention.

The ring loop of "长序列训练与上下文并行" (each rank's Q shard against the K/V
shard of rank (r - t) mod cp at ring step t, partial results merged by online
softmax) over the per-document zigzag shards of "03 · 长文负载均衡" §4.2-4.3.
The merged result, scattered back to the pack's rows, must equal unsharded
causal per-document attention (the fp64 oracle) within the method's
tolerances, in both launch schemes of the benchmark (one attention per (rank,
step) pair, or one per ring step over all ranks) and with the merges run
separately or fused into the attention epilogue.
- The 131072-token pack with cp = 8 (the benchmark's configuration): sampled
  rows -- random ones plus every document's first and last row and both sides
  of every zigzag chunk boundary.
- A ~4K-token pack with ragged documents (2cp does not divide most lengths,
  some documents are shorter than 2cp): every element.
Also: the device worklist of a ring step is bit-exact against the oracle's.
"""
import functools

import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import api
from packed_varlen_attention_cu_gb300 import workloads as W
from packed_varlen_attention_cu_gb300.ring import ZigzagRing

from gpu_util import compare, oracle_mask, to_np
from test_gpu_worklist import _assert_same, _gpu_worklist

pytestmark = pytest.mark.gpu

SCHEMES = [(True, False), (True, True), (False, False), (False, True)]
SCHEME_IDS = ["per-step", "per-step-fused", "per-pair", "per-pair-fused"]


def _run_ring(q, k, v, cu, cp, hq, hkv, d, per_step, fused):
    ring = ZigzagRing(cu, cp, hq, hkv, d, c_tile=api.default_c_tile(d), per_step=per_step,
                      fused=fused)
    ring.step(q, k, v)
    torch.cuda.synchronize()
    for wl in ring.worklists():
        assert api.worklist_error(wl) == 0
    return ring


def _pick(ring, rows, heads):
    """O [n, d] and LSE [n] of (pack row, head) jobs, read from the ring's
    rank-local blocks (test-side bookkeeping)."""
    rows_t = torch.as_tensor(rows, dtype=torch.long, device="cuda")
    heads_t = torch.as_tensor(heads, dtype=torch.long, device="cuda")
    o = torch.full((len(rows), ring.d), float("nan"), dtype=torch.float32, device="cuda")
    l = torch.full((len(rows),), float("nan"), dtype=torch.float32, device="cuda")
    for mp, bo, bl in ring.outputs():
        inv = torch.full((ring.T,), -1, dtype=torch.long, device="cuda")
        inv[mp.long()] = torch.arange(mp.numel(), device="cuda")
        loc = inv[rows_t]
        sel = loc >= 0
        o[sel] = bo[loc[sel], heads_t[sel]]
        l[sel] = bl[heads_t[sel], loc[sel]]
    return to_np(o), to_np(l)


def _chunk_boundaries(cu, cp):
    rows = []
    for a, b in zip(cu[:-1], cu[1:]):
        n, c = int(b - a), 2 * cp
        if n == 0:
            continue
        start = 0
        for ch in range(c):
            ln = n // c + (1 if ch < n % c else 0)
            if ln > 0:
                rows += [a + start, a + start + ln - 1]
            start += ln
    return rows


@functools.lru_cache(maxsize=1)
def _pack_128k():
    w = W.zigzag_pack()
    q, k, v = W.workload_qkv(w, device="cuda")
    cu = w.cu_seqlens
    special = _chunk_boundaries(cu, w.cp)
    jobs = W.random_rows(w.total_tokens, w.num_q_heads, 192, seed=23, must_include=special)
    import oracle
    jt = torch.from_numpy(jobs).long()
    qfull = torch.zeros_like(q, device="cpu")
    qfull[jt[:, 0]] = q[jt[:, 0].cuda()].cpu()
    ref_o, ref_l = oracle.attention(oracle.bf16_bits(qfull), oracle.bf16_bits(k),
                                    oracle.bf16_bits(v), cu, oracle.Mask(), jobs=jobs)
    return w, q, k, v, jobs, ref_o, ref_l


@pytest.mark.parametrize("per_step,fused", SCHEMES, ids=SCHEME_IDS)
def test_ring_cp8_128k_pack_sampled(per_step, fused):
    w, q, k, v, jobs, ref_o, ref_l = _pack_128k()
    assert w.cp == 8
    ring = _run_ring(q, k, v, w.cu_seqlens, w.cp, w.num_q_heads, w.num_kv_heads, w.head_dim,
                     per_step, fused)
    # every row of the pack sees itself: all results finite, all rows covered
    covered = 0
    for mp, bo, bl in ring.outputs():
        assert torch.isfinite(bo).all() and torch.isfinite(bl).all()
        covered += mp.numel()
    assert covered == w.total_tokens
    o, l = _pick(ring, jobs[:, 0], jobs[:, 1])
    compare(o, l, ref_o, ref_l,
            f"cp=8 ring on the 128K pack ({'step' if per_step else 'pair'}, fused={fused})")


RAGGED = [1000, 17, 333, 1500, 3, 1250, 15, 0, 7]


@pytest.mark.parametrize("per_step,fused", SCHEMES, ids=SCHEME_IDS)
@pytest.mark.parametrize("d", [64, 128])
def test_ring_cp8_ragged_pack_every_element(oracle_mod, per_step, fused, d):
    cu = W.cu_seqlens_of(RAGGED)
    T = int(cu[-1])
    hq, hkv = 4, 2
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 40 + d)
    ring = _run_ring(q.cuda(), k.cuda(), v.cuda(), cu, 8, hq, hkv, d, per_step, fused)
    rows = np.repeat(np.arange(T), hq)
    heads = np.tile(np.arange(hq), T)
    o, l = _pick(ring, rows, heads)
    o, l = o.reshape(T, hq, d), l.reshape(T, hq).T
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu, oracle_mask(W.MASK_CAUSAL))
    compare(o, l, ref_o, ref_l, f"cp=8 ragged d={d}")


@pytest.mark.parametrize("cp", [2, 8])
@pytest.mark.parametrize("dispatch", [api.DISPATCH_STATIC, api.DISPATCH_DYNAMIC])
def test_ring_step_worklist_bit_exact(oracle_mod, cp, dispatch):
    for cu in (W.tiny_pack(seed=3).cu_seqlens, W.cu_seqlens_of(RAGGED)):
        T = int(cu[-1])
        for t in range(cp):
            mask = api.make_mask(W.MASK_ZIGZAG_STEP, T, T, cp=cp, ring_step=t)
            g, counts = _gpu_worklist(cu, mask, 4, 2, 13, 7, dispatch)
            o = oracle_mod.worklist(cu, oracle_mask(W.MASK_ZIGZAG_STEP, cp=cp, ring_step=t),
                                    128, 128, 4, 2, 13, 7)
            _assert_same(g, o)
            assert counts["pairs_per_head"] == o["pairs_per_head"]


def test_ring_map_bit_exact(oracle_mod):
    for cu in (W.zigzag_pack().cu_seqlens, W.cu_seqlens_of(RAGGED)):
        T = int(cu[-1])
        for cp in (1, 3, 8):
            m = torch.full((T,), -1, dtype=torch.int32, device="cuda")
            api.zigzag_ring_map(torch.from_numpy(cu).cuda(), cp, m)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(m.cpu().numpy(), oracle_mod.ring_map(cu, cp))


@pytest.mark.parametrize("per_step,fused", SCHEMES, ids=SCHEME_IDS)
def test_ring_cp8_documents_shorter_than_the_ranks(oracle_mod, per_step, fused):
    """Documents shorter than 2cp leave some ranks without rows of them, and rank
    7 here without any row at all: its shard and every pair with it are empty."""
    lengths = [1, 5, 3, 0, 6, 2]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    assert min(api.zigzag_shard_len(cu, 8, r) for r in range(8)) == 0
    hq, hkv, d = 2, 1, 64
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 77)
    ring = _run_ring(q.cuda(), k.cuda(), v.cuda(), cu, 8, hq, hkv, d, per_step, fused)
    rows = np.repeat(np.arange(T), hq)
    heads = np.tile(np.arange(hq), T)
    o, l = _pick(ring, rows, heads)
    o, l = o.reshape(T, hq, d), l.reshape(T, hq).T
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu, oracle_mask(W.MASK_CAUSAL))
    compare(o, l, ref_o, ref_l, "cp=8, documents shorter than 2cp")
