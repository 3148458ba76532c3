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

from gpu_util import accumulate_gpu, compare, oracle_mask, run_gpu, to_np

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


def _ring(q, k, v, cu, cp, hq, hkv, d, fused=False):
    """Zigzag CP emulation: per rank, its Q shard against the KV shard of rank
    (r - t) mod cp at ring step t, partials merged left to right; the result
    is scattered back to global row order.  fused: each step merges into the
    running (O, LSE) in the attention epilogue (pva_attn_fwd_accumulate)
    instead of writing partials for pva_merge_partials."""
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
        if fused:
            # never-merged running rows may hold anything: the kernel must not read them
            acc_o = torch.full((n, hq, d), float("nan"), dtype=torch.float32, device=dev)
            acc_l = torch.full((hq, n), float("-inf"), dtype=torch.float32, device=dev)
        for t in range(cp):
            s = (r - t) % cp
            ns = maps[s].numel()
            ks = torch.empty((ns, hkv, d), dtype=torch.bfloat16, device=dev)
            vs = torch.empty_like(ks)
            api.gather_rows(k, maps[s], ks)
            api.gather_rows(v, maps[s], vs)
            mask = api.make_mask(W.MASK_ZIGZAG_PAIR, n, ns, cp=cp, q_rank=r, k_rank=s)
            if fused:
                accumulate_gpu(qr, ks, vs, cu, mask, hq, hkv, acc_o, acc_l)
                continue
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


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("cp", [2, 4])
def test_zigzag_ring_equals_unsharded(oracle_mod, cp, fused):
    lengths = [900, 5, 300, 1300, 64, 1]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    hq, hkv, d = 4, 2, 128
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 31)
    o, l = _ring(q.cuda(), k.cuda(), v.cuda(), cu, cp, hq, hkv, d, fused=fused)
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu, oracle_mask(W.MASK_CAUSAL))
    compare(to_np(o), to_np(l), ref_o, ref_l, f"ring cp={cp}")


@pytest.mark.parametrize("d", [64, 128])
def test_fused_step_matches_oracle_merge(oracle_mod, d):
    """One fused ring step = oracle merge(running, oracle attention of the step).
    The q shard of rank 0 against rank 1's kv shard has rows with no key (they
    keep the running values); running rows with LSE -inf hold NaN, which the
    kernel must not read."""
    cp, qr, kr = 2, 0, 1
    lengths = [700, 130, 1, 260]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    hq, hkv = 4, 2
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 7 + d)
    mq = oracle_mod.zigzag_map(cu, cp, qr)[0]
    mk = oracle_mod.zigzag_map(cu, cp, kr)[0]
    qs, ks, vs = q[mq], k[mk], v[mk]
    n = qs.shape[0]
    g = torch.Generator().manual_seed(d)
    o_run = torch.randn((n, hq, d), generator=g)
    l_run = torch.randn((hq, n), generator=g) * 3
    l_run[:, ::3] = -float("inf")
    o_run[::3, :, :] = float("nan")       # rows whose LSE is -inf in every head
    o_run0, l_run0 = o_run.double().numpy(), l_run.double().numpy()
    o_dev, l_dev = o_run.cuda(), l_run.cuda()
    mask = api.make_mask(W.MASK_ZIGZAG_PAIR, n, ks.shape[0], cp=cp, q_rank=qr, k_rank=kr)
    accumulate_gpu(qs, ks, vs, cu, mask, hq, hkv, o_dev, l_dev)
    so, sl = oracle_mod.attention(oracle_mod.bf16_bits(qs), oracle_mod.bf16_bits(ks),
                                  oracle_mod.bf16_bits(vs), cu,
                                  oracle_mask(W.MASK_ZIGZAG_PAIR, cp=cp, q_rank=qr, k_rank=kr))
    assert np.isneginf(sl).any() and np.isfinite(sl).any()   # both kinds of rows occur
    o_run0 = np.where(np.isneginf(l_run0).T[:, :, None], 0.0, o_run0)  # merge identity
    ro, rl = oracle_mod.merge(o_run0, l_run0, so, sl)
    got_o, got_l = to_np(o_dev), l_dev.cpu().numpy()
    # rows without keys in this step keep their running values bit for bit
    keep = np.isneginf(sl)
    np.testing.assert_array_equal(got_l[keep], l_run.numpy()[keep])
    np.testing.assert_array_equal(got_o.transpose(1, 0, 2)[keep],
                                  o_run.double().numpy().transpose(1, 0, 2)[keep])
    # where nothing was ever merged (LSE still -inf) O is the untouched running value
    empty = np.isneginf(rl).T[:, :, None]
    compare(np.where(empty, 0.0, got_o), got_l, ro, rl, f"fused step d={d}")
