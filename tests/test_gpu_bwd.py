"""Backward on the GPU against the fp64 oracle: dq, dk, dv element by element
(relative L2 and max-abs against the gradient's scale), for document-causal,
sliding-window, zigzag-pair and explicit-slice masks, GQA, d = 64 and 128,
bf16 and fp32 gradients, ragged documents."""
import ctypes

import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import api
from packed_varlen_attention_cu_gb300 import workloads as W

from gpu_util import oracle_mask, run_gpu

pytestmark = pytest.mark.gpu

# bf16 P and dS (2^-9 relative rounding per term) feed the gradient MMAs; measured
# 1.5-2.6e-3 relative L2 and at most 3.8e-3 of the largest magnitude
REL_L2 = 6e-3
MAX_ABS_REL = 1.5e-2   # of the largest reference magnitude


def _bwd(q, k, v, cu, mask, hq, hkv, dout, fp32):
    dev = torch.device("cuda")
    out, lse, wl = run_gpu(q, k, v, cu, mask, hq, hkv)
    nd = len(cu) - 1
    params = api.make_params(hq, hkv)
    plan = api.alloc_bwd_plan(nd, mask, params, dev)
    api.build_bwd_plan(wl, nd, mask, params, plan)
    dt = torch.float32 if fp32 else torch.bfloat16
    dq = torch.full(q.shape, float("nan"), dtype=dt, device=dev)
    dk = torch.full(k.shape, float("nan"), dtype=dt, device=dev)
    dv = torch.full(v.shape, float("nan"), dtype=dt, device=dev)
    cu_d = torch.from_numpy(np.ascontiguousarray(cu, dtype=np.int32)).to(dev)
    api.attn_bwd(q.to(dev), k.to(dev), v.to(dev), out, lse, dout.to(dev), cu_d, nd, mask, params,
                 wl, plan, dq, dk, dv)
    torch.cuda.synchronize()
    assert api.worklist_error(wl) == 0
    return [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]


def _check(got, ref, label):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(g).all(), f"{label} {name}: non-finite"
        scale = max(float(np.abs(r).max()), 1e-6)
        err = np.abs(g - r)
        rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-12))
        msg = f"{label} {name}: rel_l2={rel:.3e} max_abs/scale={err.max() / scale:.3e}"
        print(msg)
        assert rel <= REL_L2, msg
        assert err.max() <= MAX_ABS_REL * scale, msg


def _case(oracle_mod, lengths, hq, hkv, d, kind, fp32, seed, **mkw):
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, T, hq, hkv, d, seed)
    dout = W.make_qkv(T, T, hq, hkv, d, seed + 100)[0]
    mask = api.make_mask(kind, T, T, **mkw)
    okw = {"window": mkw.get("window", 0), "num_prefix": mkw.get("num_prefix_docs", 0)}
    got = _bwd(q, k, v, cu, mask, hq, hkv, dout, fp32)
    ref = oracle_mod.attention_bwd(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                   oracle_mod.bf16_bits(v), oracle_mod.bf16_bits(dout), cu,
                                   oracle_mask(kind, **okw))
    _check(got, ref, f"{kind} d={d} hq={hq}/{hkv} fp32={fp32}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("fp32", [True, False])
def test_bwd_causal_gqa(oracle_mod, d, fp32):
    _case(oracle_mod, [300, 5, 130, 700, 1, 129], 4, 2, d, W.MASK_CAUSAL, fp32, 21)


def test_bwd_causal_mha_long_doc(oracle_mod):
    _case(oracle_mod, [1500, 37], 2, 2, 128, W.MASK_CAUSAL, True, 22)


def test_bwd_sliding_window(oracle_mod):
    _case(oracle_mod, [900, 250, 64], 4, 1, 128, W.MASK_SLIDING_WINDOW, True, 23, window=200)


def test_bwd_zigzag_pair(oracle_mod):
    cp, qr, kr = 2, 1, 0
    lengths = [700, 130, 1, 260]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    hq, hkv, d = 4, 2, 128
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 24)
    dout = W.make_qkv(T, T, hq, hkv, d, 124)[0]
    mq = oracle_mod.zigzag_map(cu, cp, qr)[0]
    mk = oracle_mod.zigzag_map(cu, cp, kr)[0]
    qs, ks, vs, ds = q[mq], k[mk], v[mk], dout[mq]
    mask = api.make_mask(W.MASK_ZIGZAG_PAIR, qs.shape[0], ks.shape[0], cp=cp, q_rank=qr, k_rank=kr)
    got = _bwd(qs, ks, vs, cu, mask, hq, hkv, ds, True)
    ref = oracle_mod.attention_bwd(oracle_mod.bf16_bits(qs), oracle_mod.bf16_bits(ks),
                                   oracle_mod.bf16_bits(vs), oracle_mod.bf16_bits(ds), cu,
                                   oracle_mask(W.MASK_ZIGZAG_PAIR, cp=cp, q_rank=qr, k_rank=kr))
    _check(got, ref, "zigzag pair")


def test_bwd_explicit_slices_with_unseen_keys(oracle_mod):
    # queries [0, 300) see keys [0, 200) causally and queries [300, 420) see keys
    # [250, 400) fully; keys [200, 250) and [400, 450) are never seen (zero gradient)
    sl = np.array([[0, 300, 0, 0, 200, 0, 1, 0], [300, 120, 0, 250, 150, 0, 0, 0]], dtype=np.int32)
    Tq, Tk, hq, hkv, d = 420, 450, 2, 1, 64
    q, _, _ = W.make_qkv(Tq, Tq, hq, hkv, d, 25)
    _, k, v = W.make_qkv(Tk, Tk, hq, hkv, d, 26)
    dout = W.make_qkv(Tq, Tq, hq, hkv, d, 27)[0]
    mask = api.make_mask(W.MASK_SLICES, Tq, Tk, slices=sl)
    cu = W.cu_seqlens_of([Tq])
    got = _bwd(q, k, v, cu, mask, hq, hkv, dout, True)
    ref = oracle_mod.attention_bwd(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                   oracle_mod.bf16_bits(v), oracle_mod.bf16_bits(dout), cu,
                                   oracle_mask(W.MASK_SLICES, slices=sl))
    _check(got, ref, "slices")
    assert np.all(got[1][200:250] == 0) and np.all(got[2][400:] == 0)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_inv_and_bi_causal_slices(oracle_mod, d):
    # INV-CAUSAL, BI-CAUSAL, windowed CAUSAL and FULL slices over three key ranges
    # (identical or disjoint, as the backward plan requires)
    sl = np.array([[0, 300, 0, 0, 300, 0, 2, 0],
                   [300, 200, 1000, 300, 300, 1000, 3, 0],
                   [300, 200, 1000, 0, 300, 900, 1, 64],
                   [500, 400, 0, 600, 300, 50, 2, 200],
                   [500, 400, 0, 300, 300, 0, 0, 0]], dtype=np.int32)
    T, hq, hkv = 900, 4, 2
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 50 + d)
    dout = W.make_qkv(T, T, hq, hkv, d, 150 + d)[0]
    mask = api.make_mask(W.MASK_SLICES, T, T, slices=sl)
    cu = W.cu_seqlens_of([T])
    got = _bwd(q, k, v, cu, mask, hq, hkv, dout, True)
    ref = oracle_mod.attention_bwd(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                   oracle_mod.bf16_bits(v), oracle_mod.bf16_bits(dout), cu,
                                   oracle_mask(W.MASK_SLICES, slices=sl))
    _check(got, ref, f"inv/bi slices d={d}")


def test_bwd_shared_question(oracle_mod):
    # the question's keys form one key group: its own causal slice and every answer
    _case(oracle_mod, [400, 300, 200, 129], 4, 2, 128, W.MASK_SHARED_QUESTION, True, 28,
          num_prefix_docs=1)


def test_bwd_plan_rejects_partly_overlapping_key_ranges():
    sl = np.array([[0, 10, 0, 0, 10, 0, 1, 0], [10, 10, 0, 5, 10, 0, 0, 0]], dtype=np.int32)
    m = api.make_mask(W.MASK_SLICES, 20, 20, slices=sl)
    p = api.make_params(2, 2)
    assert api.lib().pva_bwd_plan_bytes(1, ctypes.byref(m), ctypes.byref(p)) == 0


@pytest.mark.parametrize("wname", ["zigzag_pack", "long_tail_gqa"])
def test_bwd_full_workload_sampled(oracle_mod, wname):
    """The bench's configurations: the 128K causal pack (32 q / 8 kv heads, d = 128)
    and the eight long-tail GQA packs (14 q / 2 kv heads, d = 64: three S^T/dP^T
    buffers, warpgroups on alternate half-items), bf16 gradients: sampled dq rows
    and dk/dv keys against the oracle, each by definition."""
    w = getattr(W, wname)()
    cu = w.cu_seqlens
    T, hq, hkv, d = w.total_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    q, k, v = W.workload_qkv(w, device="cpu")
    dout = W.make_qkv(T, T, hq, hkv, d, w.seed + 1000)[0]
    mask = api.mask_for_workload(w)
    got = _bwd(q, k, v, cu, mask, hq, hkv, dout, False)
    rng = np.random.default_rng(7)
    lens = np.diff(cu)
    qj = np.stack([rng.integers(0, T, 48), rng.integers(0, hq, 48)], axis=1)
    # keys: random ones, plus the first and last key of the longest document
    big = int(np.argmax(lens))
    kj = np.stack([rng.integers(0, T, 14), rng.integers(0, hkv, 14)], axis=1)
    kj = np.concatenate([kj, [[cu[big], 0], [cu[big + 1] - 1, hkv - 1]]])
    bits = [oracle_mod.bf16_bits(x) for x in (q, k, v, dout)]
    rq, rk, rv = oracle_mod.attention_bwd_jobs(*bits, cu, oracle_mask(W.MASK_CAUSAL), qj, kj)
    gq = got[0][qj[:, 0], qj[:, 1]]
    gk = got[1][kj[:, 0], kj[:, 1]]
    gv = got[2][kj[:, 0], kj[:, 1]]
    _check((gq, gk, gv), (rq, rk, rv), f"{wname} sampled")


@pytest.mark.parametrize("t", [0, 1, 3])
def test_bwd_zigzag_ring_step(oracle_mod, t):
    """One ring step of every rank at once (PVA_MASK_ZIGZAG_STEP, Q/K/V in ring
    order): key chunks that no query of their step sees get a zero gradient."""
    cp = 4
    lengths = [700, 130, 1, 260, 33]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    hq, hkv, d = 4, 2, 128
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 60 + t)
    dout = W.make_qkv(T, T, hq, hkv, d, 160 + t)[0]
    ring = oracle_mod.ring_map(cu, cp)
    qs, ks, vs, ds = q[ring], k[ring], v[ring], dout[ring]
    mask = api.make_mask(W.MASK_ZIGZAG_STEP, T, T, cp=cp, ring_step=t)
    got = _bwd(qs, ks, vs, cu, mask, hq, hkv, ds, True)
    ref = oracle_mod.attention_bwd(oracle_mod.bf16_bits(qs), oracle_mod.bf16_bits(ks),
                                   oracle_mod.bf16_bits(vs), oracle_mod.bf16_bits(ds), cu,
                                   oracle_mask(W.MASK_ZIGZAG_STEP, cp=cp, ring_step=t))
    _check(got, ref, f"ring step t={t}")


def _bwd_with(q, k, v, cu, mask, params, dout):
    """Forward and backward with explicit worklist params; bf16 gradients on the device."""
    dev = torch.device("cuda")
    nd = len(cu) - 1
    cu_d = torch.from_numpy(np.ascontiguousarray(cu, dtype=np.int32)).to(dev)
    wl = api.alloc_worklist(nd, mask, params, dev)
    api.build_worklist(cu_d, mask, params, wl)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=dev)
    api.attn_fwd(qd, kd, vd, cu_d, mask, params, wl, out, lse)
    plan = api.alloc_bwd_plan(nd, mask, params, dev)
    api.build_bwd_plan(wl, nd, mask, params, plan)
    grads = [torch.full(t.shape, float("nan"), dtype=torch.bfloat16, device=dev) for t in (q, k, v)]
    api.attn_bwd(qd, kd, vd, out, lse, dout.to(dev), cu_d, nd, mask, params, wl, plan, *grads)
    torch.cuda.synchronize()
    assert api.worklist_error(wl) == 0
    return grads


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("num_ctas", [0, 5])
def test_bwd_bitwise_equal_across_dispatch(num_ctas, d):
    # Each gradient row is summed by one CTA in an order fixed by its unit (dQ: the
    # forward unit's kv tiles; dK/dV: the plan unit's q tiles and heads), so the
    # dispatch mode and the CTA count change who computes a row, never its value
    # (at d = 64 they also change which element-wise warpgroup takes a half-item).
    lengths = [300, 1, 777, 128, 0, 64, 1500, 129]
    hq, hkv = 8, 2
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 5)
    dout = W.make_qkv(T, T, hq, hkv, d, 105)[0]
    mask = api.make_mask(W.MASK_CAUSAL, T, T)
    runs = [_bwd_with(q, k, v, cu, mask, api.make_params(hq, hkv, num_ctas=num_ctas, dispatch=dp),
                      dout)
            for dp in (api.DISPATCH_DYNAMIC, api.DISPATCH_STATIC)]
    for name, a, b in zip(("dq", "dk", "dv"), *runs):
        assert torch.isfinite(a.float()).all(), name
        assert torch.equal(a, b), name


def test_bwd_static_dispatch_matches_oracle(oracle_mod):
    lengths = [200, 513, 7, 300]
    hq, hkv, d = 4, 2, 64
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, T, hq, hkv, d, 11)
    dout = W.make_qkv(T, T, hq, hkv, d, 111)[0]
    mask = api.make_mask(W.MASK_CAUSAL, T, T)
    got = _bwd_with(q, k, v, cu, mask,
                    api.make_params(hq, hkv, num_ctas=3, dispatch=api.DISPATCH_STATIC), dout)
    ref = oracle_mod.attention_bwd(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                   oracle_mod.bf16_bits(v), oracle_mod.bf16_bits(dout), cu,
                                   oracle_mask(W.MASK_CAUSAL))
    _check([t.float().cpu().numpy().astype(np.float64) for t in got], ref, "static dispatch")
