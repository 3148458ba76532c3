"""Short documents sharing tiles (pva_worklist_params.pack_docs) on the GPU.

"03 · 长文负载均衡" §4.1: a block shorter than a tile is still charged as a
whole tile.  With pack_docs = 1 consecutive documents shorter than a tile are
grouped into one query tile against one key tile, each row masked to its own
document.  The forward and the backward must still equal the fp64 oracle's
per-document attention (which knows nothing of the packing) at the method's
tolerances, and the packed worklist must compute fewer tiles.
"""
import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import api
from packed_varlen_attention_cu_gb300 import workloads as W

from gpu_util import compare, oracle_mask, run_gpu, to_np
from test_gpu_bwd import _check

pytestmark = pytest.mark.gpu

SHORT = [5, 130, 1, 9, 0, 12, 3, 128, 40, 40, 40, 8, 15, 127, 1, 64, 64, 2, 250]


def _fwd_case(oracle_mod, lengths, hq, hkv, d, kind, window, seed, dispatch, out_fp32=False):
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, T, hq, hkv, d, seed)
    mask = api.make_mask(kind, T, T, window=window)
    out, lse, wl = run_gpu(q, k, v, cu, mask, hq, hkv, c_tile=api.default_c_tile(d),
                           out_fp32=out_fp32, dispatch=dispatch, pack_docs=1)
    g = api.decode_worklist(wl)
    assert g["pack_docs"] == 1 and (g["slices"][:, 6] == 4).any()
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu, oracle_mask(kind, window))
    compare(to_np(out), to_np(lse), ref_o, ref_l, f"packed {kind} d={d} {hq}/{hkv}")
    return wl


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (6, 2), (7, 1)])
@pytest.mark.parametrize("dispatch", [api.DISPATCH_DYNAMIC, api.DISPATCH_STATIC])
def test_packed_forward_causal(oracle_mod, d, hq, hkv, dispatch):
    _fwd_case(oracle_mod, SHORT * 3, hq, hkv, d, W.MASK_CAUSAL, 0, 50 + d + hq, dispatch)


@pytest.mark.parametrize("window", [1, 7, 100])
def test_packed_forward_window(oracle_mod, window):
    _fwd_case(oracle_mod, SHORT * 2, 4, 2, 128, W.MASK_SLIDING_WINDOW, window, 60 + window,
              api.DISPATCH_DYNAMIC)


def test_packed_forward_fp32_partials_and_equal_to_unpacked(oracle_mod):
    lengths = [3, 4, 5, 6, 7, 8, 9, 10, 11, 12] * 8
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, T, 4, 2, 64, 70)
    mask = api.make_mask(W.MASK_CAUSAL, T, T)
    o_p, l_p, wl_p = run_gpu(q, k, v, cu, mask, 4, 2, out_fp32=True, pack_docs=1)
    o_u, l_u, wl_u = run_gpu(q, k, v, cu, mask, 4, 2, out_fp32=True, pack_docs=0)
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu, oracle_mask(W.MASK_CAUSAL))
    compare(to_np(o_p), to_np(l_p), ref_o, ref_l, "packed fp32")
    cp_, cu_ = api.worklist_counts(wl_p), api.worklist_counts(wl_u)
    assert cp_["pairs_per_head"] == cu_["pairs_per_head"]
    assert cp_["tiles_per_head"] < cu_["tiles_per_head"] and cp_["units"] < cu_["units"]


@pytest.mark.parametrize("d", [64, 128])
def test_packed_backward(oracle_mod, d):
    lengths = SHORT * 2
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    hq, hkv = 4, 2
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 80 + d)
    dout = W.make_qkv(T, T, hq, hkv, d, 180 + d)[0]
    dev = torch.device("cuda")
    mask = api.make_mask(W.MASK_CAUSAL, T, T)
    out, lse, wl = run_gpu(q, k, v, cu, mask, hq, hkv, pack_docs=1)
    nd = len(lengths)
    params = api.make_params(hq, hkv, pack_docs=1)
    plan = api.alloc_bwd_plan(nd, mask, params, dev)
    api.build_bwd_plan(wl, nd, mask, params, plan)
    dq = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
    dk = torch.full(k.shape, float("nan"), dtype=torch.float32, device=dev)
    dv = torch.full(v.shape, float("nan"), dtype=torch.float32, device=dev)
    api.attn_bwd(q.to(dev), k.to(dev), v.to(dev), out, lse, dout.to(dev),
                 torch.from_numpy(cu).to(dev), nd, mask, params, wl, plan, dq, dk, dv)
    torch.cuda.synchronize()
    assert api.worklist_error(wl) == 0
    got = [t.cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]
    ref = oracle_mod.attention_bwd(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                   oracle_mod.bf16_bits(v), oracle_mod.bf16_bits(dout), cu,
                                   oracle_mask(W.MASK_CAUSAL))
    _check(got, ref, f"packed backward d={d}")


def test_packed_long_tail_full_size_sampled(oracle_mod):
    """The 8-pack long-tail workload with packing, sampled rows (each document's
    first and last row included) against the oracle."""
    w = W.long_tail_gqa()
    cu = w.cu_seqlens
    T = w.total_tokens
    q, k, v = W.workload_qkv(w, device="cuda")
    mask = api.mask_for_workload(w)
    out, lse, _ = run_gpu(q, k, v, cu, mask, w.num_q_heads, w.num_kv_heads,
                          c_tile=api.default_c_tile(w.head_dim), pack_docs=1)
    special = []
    for a, b in zip(cu[:-1], cu[1:]):
        if b > a:
            special += [a, b - 1]
    jobs = W.random_rows(T, w.num_q_heads, 192, seed=29, must_include=special)
    jt = torch.from_numpy(jobs).long()
    qfull = torch.zeros((T, w.num_q_heads, w.head_dim), dtype=torch.bfloat16)
    qfull[jt[:, 0]] = q[jt[:, 0].cuda()].cpu()
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(qfull), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu, oracle_mask(W.MASK_CAUSAL),
                                        jobs=jobs)
    got_o = to_np(out[jt[:, 0].cuda(), jt[:, 1].cuda()])
    got_l = to_np(lse[jt[:, 1].cuda(), jt[:, 0].cuda()])
    compare(got_o, got_l, ref_o, ref_l, "long-tail packed")
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
