"""Merge, zigzag maps, gather and the zigzag ring emulation on the GPU.

"03 · 长文负载均衡" §3.2 (online-softmax rescale-and-sum of partials) and
§4.2-4.3 (zigzag per document); the ring loop of "长序列训练与上下文并行"
(each rank's Q against every KV shard in ring order, merged step by step).
"""
import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import api
from packed_varlen_attention_cu_gb300 import workloads as W

from gpu_util import compare, oracle_mask, run_gpu, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cp", [1, 2, 3, 8])
def test_zigzag_maps_bit_exact(oracle_mod, cp):
    w = W.zigzag_pack()
    cu = w.cu_seqlens
    cu_d = torch.from_numpy(cu).cuda()
    for r in range(cp):
        n = api.zigzag_shard_len(cu, cp, r)
        ref_map, ref_table = oracle_mod.zigzag_map(cu, cp, r)
        assert n == ref_map.shape[0]
        gmap = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        table = torch.zeros((w.num_docs, 2, 4), dtype=torch.int32, device="cuda")
        api.zigzag_shard(cu_d, cp, r, gmap, table)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(gmap.cpu().numpy(), ref_map)
        np.testing.assert_array_equal(table.cpu().numpy(), ref_table)


def test_zigzag_maps_empty_and_short_docs(oracle_mod):
    cu = W.cu_seqlens_of([0, 1, 5, 0, 17, 2, 0])
    cu_d = torch.from_numpy(cu).cuda()
    for cp in (1, 4):
        for r in range(cp):
            n = api.zigzag_shard_len(cu, cp, r)
            gmap = torch.full((max(n, 1),), -1, dtype=torch.int32, device="cuda")
            api.zigzag_shard(cu_d, cp, r, gmap)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(gmap.cpu().numpy()[:n], oracle_mod.zigzag_map(cu, cp, r)[0])


@pytest.mark.parametrize("fp32", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_merge_matches_oracle(oracle_mod, fp32, d):
    g = torch.Generator().manual_seed(d + fp32)
    t, h = 1000, 6
    dt = torch.float32 if fp32 else torch.bfloat16
    oa = torch.randn((t, h, d), generator=g).to(dt)
    ob = torch.randn((t, h, d), generator=g).to(dt)
    la = torch.randn((h, t), generator=g) * 4
    lb = torch.randn((h, t), generator=g) * 4
    la[0, :7] = -float("inf")
    lb[0, 3:9] = -float("inf")
    out = torch.empty((t, h, d), dtype=dt, device="cuda")
    lo = torch.empty((h, t), dtype=torch.float32, device="cuda")
    api.merge_partials(oa.cuda(), la.cuda(), ob.cuda(), lb.cuda(), out, lo)
    torch.cuda.synchronize()
    ro, rl = oracle_mod.merge(oa.double().numpy(), la.double().numpy(), ob.double().numpy(),
                              lb.double().numpy())
    tol = 1e-5 if fp32 else 1e-2
    np.testing.assert_allclose(to_np(out), ro, atol=tol, rtol=tol)
    np.testing.assert_array_equal(np.isneginf(lo.cpu().numpy()), np.isneginf(rl))
    fin = np.isfinite(rl)
    np.testing.assert_allclose(lo.cpu().numpy()[fin], rl[fin], atol=1e-5, rtol=1e-6)


def test_merge_in_place_and_identity():
    t, h, d = 513, 4, 128
    oa = torch.randn((t, h, d), device="cuda")
    la = torch.randn((h, t), device="cuda")
    ob = torch.randn((t, h, d), device="cuda")
    lb = torch.full((h, t), -float("inf"), device="cuda")
    keep_o, keep_l = oa.clone(), la.clone()
    api.merge_partials(oa, la, ob, lb, oa, la)  # in place, b carries nothing
    torch.cuda.synchronize()
    torch.testing.assert_close(oa, keep_o, atol=1e-6, rtol=1e-6)
    torch.testing.assert_close(la, keep_l, atol=1e-6, rtol=1e-6)


def test_gather_scatter_roundtrip():
    src = torch.randn((1000, 8, 64), device="cuda").to(torch.bfloat16)
    perm = torch.randperm(1000, device="cuda").to(torch.int32)
    dst = torch.empty_like(src)
    api.gather_rows(src, perm, dst)
    back = torch.empty_like(src)
    api.gather_rows(dst, perm, back, scatter=True)
    torch.cuda.synchronize()
    assert torch.equal(dst, src[perm.long()]) and torch.equal(back, src)
    # out-of-range map entries are skipped, never dereferenced
    bad = perm.clone()
    bad[:5] = 5000
    dst2 = torch.zeros_like(src)
    api.gather_rows(src, bad, dst2)
    torch.cuda.synchronize()
    assert torch.all(dst2[:5] == 0) and torch.equal(dst2[5:], src[perm[5:].long()])


def _ring(q, k, v, cu, cp, hq, hkv, d):
    """Zigzag CP emulation: per rank, its Q shard against the KV shard of rank
    (r - t) mod cp at ring step t, partials merged left to right; the result
    is scattered back to global row order."""
    dev = torch.device("cuda")
    T = q.shape[0]
    cu_d = torch.from_numpy(cu).to(dev)
    maps = []
    for r in range(cp):
        n = api.zigzag_shard_len(cu, cp, r)
        m = torch.empty((n,), dtype=torch.int32, device=dev)
        api.zigzag_shard(cu_d, cp, r, m)
        maps.append(m)
    o_full = torch.empty((T, hq, d), dtype=torch.float32, device=dev)
    l_full = torch.empty((hq, T), dtype=torch.float32, device=dev)
    for r in range(cp):
        n = maps[r].numel()
        qr = torch.empty((n, hq, d), dtype=torch.bfloat16, device=dev)
        api.gather_rows(q, maps[r], qr)
        acc_o = acc_l = None
        for t in range(cp):
            s = (r - t) % cp
            ns = maps[s].numel()
            ks = torch.empty((ns, hkv, d), dtype=torch.bfloat16, device=dev)
            vs = torch.empty_like(ks)
            api.gather_rows(k, maps[s], ks)
            api.gather_rows(v, maps[s], vs)
            mask = api.make_mask(W.MASK_ZIGZAG_PAIR, n, ns, cp=cp, q_rank=r, k_rank=s)
            o, l, _ = run_gpu(qr, ks, vs, cu, mask, hq, hkv, out_fp32=True)
            if acc_o is None:
                acc_o, acc_l = o, l
            else:
                api.merge_partials(acc_o, acc_l, o, l, acc_o, acc_l)
        api.gather_rows(acc_o, maps[r], o_full, scatter=True)
        # LSE is [heads, tokens]: scatter per head row
        for h in range(hq):
            l_full[h, maps[r].long()] = acc_l[h]
    torch.cuda.synchronize()
    return o_full, l_full


@pytest.mark.parametrize("cp", [2, 4])
def test_zigzag_ring_equals_unsharded(oracle_mod, cp):
    lengths = [900, 5, 300, 1300, 64, 1]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    hq, hkv, d = 4, 2, 128
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 31)
    o, l = _ring(q.cuda(), k.cuda(), v.cuda(), cu, cp, hq, hkv, d)
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu, oracle_mask(W.MASK_CAUSAL))
    compare(to_np(o), to_np(l), ref_o, ref_l, f"ring cp={cp}")
