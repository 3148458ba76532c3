"""Device worklist vs the oracle's sequential worklist: bit-exact.

"03 · 长文负载均衡" §3.2 (pair-exact tile costs; only non-empty blocks) and
§2.1 / "数据并行负载均衡" §4.4 (LPT).  Every field is compared: slices,
segments, units in CTA order (with costs and pair counts), kv-tile runs and
the per-CTA CSR offsets.
"""
import numpy as np
import pytest
import torch

import oracle
from packed_varlen_attention_cu_gb300 import api
from packed_varlen_attention_cu_gb300 import workloads as W

from gpu_util import oracle_mask

pytestmark = pytest.mark.gpu


def _gpu_worklist(cu_np, mask, hq, hkv, num_ctas, c_tile, dispatch=api.DISPATCH_STATIC,
                  pack_docs=0):
    dev = torch.device("cuda")
    cu = torch.from_numpy(np.ascontiguousarray(cu_np, dtype=np.int32)).to(dev)
    params = api.make_params(hq, hkv, num_ctas=num_ctas, c_tile=c_tile, dispatch=dispatch,
                             pack_docs=pack_docs)
    wl = api.alloc_worklist(cu.numel() - 1, mask, params, dev)
    api.build_worklist(cu, mask, params, wl)
    torch.cuda.synchronize()
    assert api.worklist_error(wl) == 0
    return api.decode_worklist(wl), api.worklist_counts(wl)


def _assert_same(g, o):
    """A static worklist equals the oracle's (units in CTA order, CSR offsets);
    a dynamic one has the same units in uid order without CTAs, and its
    dispatch order is oracle.dispatch_order of the costs by uid."""
    ou = o["units"].reshape(-1, 10)
    oc, op = o["unit_cost"], o["unit_pairs"]
    if g["dispatch_order"] is not None:
        by_uid = np.argsort(ou[:, 0], kind="stable")
        ou, oc, op = ou[by_uid].copy(), oc[by_uid], op[by_uid]
        ou[:, 9] = -1
        np.testing.assert_array_equal(g["dispatch_order"],
                                      oracle.dispatch_order(oc, g["header"]["num_ctas"]))
        assert g["cta_off"] is None
    else:
        np.testing.assert_array_equal(g["cta_off"], o["cta_off"])
    np.testing.assert_array_equal(g["slices"], o["slices"].reshape(-1, 8))
    packed = o["slices"].reshape(-1, 8)[:, 6] == 4  # short documents sharing a tile
    np.testing.assert_array_equal(g["slice_masks"][packed], o["slice_masks"][packed])
    np.testing.assert_array_equal(g["segs"][:, :5], o["segs"].reshape(-1, 5))
    np.testing.assert_array_equal(g["units"], ou)
    np.testing.assert_array_equal(g["unit_cost"], oc)
    np.testing.assert_array_equal(g["unit_pairs"], op)
    np.testing.assert_array_equal(g["runs"], o["runs"].reshape(-1, 3))


CASES = [
    ("tiny", lambda: W.tiny_pack(), {}),
    ("long-tail 2 packs GQA 7:1", lambda: W.long_tail_gqa(2), {}),
    ("libra pair", lambda: W.libra_pair(), {}),
    ("shared question", lambda: W.shared_question(), {}),
    ("sliding window", lambda: W.sliding_window(), {}),
    ("128K pack", lambda: W.zigzag_pack(), {}),
]


@pytest.mark.parametrize("name,mk,kw", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("num_ctas,c_tile", [(152, 0), (148, 4096), (7, 1)])
@pytest.mark.parametrize("dispatch", [api.DISPATCH_STATIC, api.DISPATCH_DYNAMIC])
def test_worklist_bit_exact(oracle_mod, name, mk, kw, num_ctas, c_tile, dispatch):
    w = mk()
    cu = w.cu_seqlens
    mask = api.mask_for_workload(w)
    g, counts = _gpu_worklist(cu, mask, w.num_q_heads, w.num_kv_heads, num_ctas, c_tile,
                              dispatch)
    o = oracle_mod.worklist(cu, oracle_mask(w.mask_kind, w.window, w.num_prefix_docs), 128, 128,
                            w.num_q_heads, w.num_kv_heads, num_ctas, c_tile)
    _assert_same(g, o)
    assert counts["pairs_per_head"] == o["pairs_per_head"]


def test_worklist_pair_count_matches_closed_form():
    w = W.zigzag_pack()
    mask = api.mask_for_workload(w)
    _, counts = _gpu_worklist(w.cu_seqlens, mask, 32, 8, 152, 0)
    assert counts["pairs_per_head"] == sum(l * (l + 1) // 2 for l in w.lengths) == 488185982


@pytest.mark.parametrize("cp,c_tile", [(2, 7), (8, 7), (8, 0)])
def test_worklist_zigzag_pairs_bit_exact(oracle_mod, cp, c_tile):
    w = W.tiny_pack(seed=3)
    cu = w.cu_seqlens
    for r in range(cp):
        tq = api.zigzag_shard_len(cu, cp, r)
        for s in range(cp):
            tk = api.zigzag_shard_len(cu, cp, s)
            mask = api.make_mask(W.MASK_ZIGZAG_PAIR, tq, tk, cp=cp, q_rank=r, k_rank=s)
            g, _ = _gpu_worklist(cu, mask, 4, 2, 13, c_tile)
            o = oracle_mod.worklist(cu, oracle_mask(W.MASK_ZIGZAG_PAIR, cp=cp, q_rank=r, k_rank=s),
                                    128, 128, 4, 2, 13, c_tile)
            _assert_same(g, o)


def test_worklist_explicit_slices_bit_exact(oracle_mod):
    sl = np.array([[0, 300, 0, 0, 300, 0, 1, 0],
                   [300, 200, 1000, 0, 150, 0, 0, 0],
                   [300, 200, 1000, 300, 400, 900, 1, 64],
                   [700, 5, 0, 700, 5, 0, 1, 0]], dtype=np.int32)
    mask = api.make_mask(W.MASK_SLICES, 705, 705, slices=sl)
    g, _ = _gpu_worklist(np.array([0, 705], dtype=np.int32), mask, 2, 1, 5, 0)
    o = oracle_mod.worklist(np.array([0, 705], dtype=np.int32), oracle_mask(W.MASK_SLICES, slices=sl),
                            128, 128, 2, 1, 5, 0)
    _assert_same(g, o)


# INV-CAUSAL and BI-CAUSAL slices ("03 · 长文负载均衡" §4.4), mixed with CAUSAL and
# FULL, over three query segments and three key ranges
SLICE_TYPES_CASE = np.array([[0, 300, 0, 0, 300, 0, 2, 0],
                             [300, 200, 1000, 300, 300, 1000, 3, 0],
                             [300, 200, 1000, 0, 300, 900, 1, 64],
                             [500, 400, 0, 600, 300, 50, 2, 200],
                             [500, 400, 0, 300, 300, 0, 0, 0]], dtype=np.int32)


def test_worklist_inv_bi_causal_slices_bit_exact(oracle_mod):
    sl = SLICE_TYPES_CASE
    mask = api.make_mask(W.MASK_SLICES, 900, 900, slices=sl)
    g, _ = _gpu_worklist(np.array([0, 900], dtype=np.int32), mask, 4, 2, 7, 0)
    o = oracle_mod.worklist(np.array([0, 900], dtype=np.int32), oracle_mask(W.MASK_SLICES, slices=sl),
                            128, 128, 4, 2, 7, 0)
    _assert_same(g, o)


def test_worklist_edge_lengths_bit_exact(oracle_mod):
    lengths = [0, 1, 127, 128, 129, 0, 255, 256, 257, 1, 1, 383, 0]
    cu = W.cu_seqlens_of(lengths)
    for hq, hkv in ((1, 1), (3, 1), (6, 2), (8, 8)):
        mask = api.make_mask(W.MASK_CAUSAL, int(cu[-1]), int(cu[-1]))
        for nc in (1, 3, 1024):
            g, _ = _gpu_worklist(cu, mask, hq, hkv, nc, 11)
            o = oracle_mod.worklist(cu, oracle_mask(W.MASK_CAUSAL), 128, 128, hq, hkv, nc, 11)
            _assert_same(g, o)


def test_worklist_is_deterministic():
    w = W.long_tail_gqa(1)
    mask = api.mask_for_workload(w)
    a, _ = _gpu_worklist(w.cu_seqlens, mask, 14, 2, 152, 0)
    b, _ = _gpu_worklist(w.cu_seqlens, mask, 14, 2, 152, 0)
    for key in ("units", "unit_cost", "runs", "cta_off"):
        np.testing.assert_array_equal(a[key], b[key])


def test_bad_cu_seqlens_sets_error_not_fault():
    dev = torch.device("cuda")
    cu = torch.tensor([0, 10, 5, 20], dtype=torch.int32, device=dev)  # decreasing
    mask = api.make_mask(W.MASK_CAUSAL, 20, 20)
    params = api.make_params(2, 2, num_ctas=4)
    wl = api.alloc_worklist(3, mask, params, dev)
    api.build_worklist(cu, mask, params, wl)
    torch.cuda.synchronize()
    assert api.worklist_error(wl) != 0
    # attention on a failed worklist writes nothing and leaves the error in place
    q = torch.zeros((20, 2, 64), dtype=torch.bfloat16, device=dev)
    out = torch.full((20, 2, 64), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((2, 20), 7.0, dtype=torch.float32, device=dev)
    api.attn_fwd(q, q, q, cu, mask, params, wl, out, lse)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)


def test_worklist_single_cta_and_zero_costs(oracle_mod):
    # one bin: every unit lands on CTA 0 in cost order; zero-cost units (c_tile = 0,
    # query chunks with no key in the shard) exercise the run step of the LPT
    w = W.zigzag_pack()
    cu = w.cu_seqlens
    tq = api.zigzag_shard_len(cu, 8, 0)
    tk = api.zigzag_shard_len(cu, 8, 7)
    mask = api.make_mask(W.MASK_ZIGZAG_PAIR, tq, tk, cp=8, q_rank=0, k_rank=7)
    for nc in (1, 152):
        g, _ = _gpu_worklist(cu, mask, 32, 8, nc, 0)
        o = oracle_mod.worklist(cu, oracle_mask(W.MASK_ZIGZAG_PAIR, cp=8, q_rank=0, k_rank=7),
                                128, 128, 32, 8, nc, 0)
        _assert_same(g, o)


REFINE_CASES = [
    ("tiny", lambda: W.tiny_pack()),
    ("shared question", lambda: W.shared_question()),
    ("libra pair", lambda: W.libra_pair()),
    ("long-tail 2 packs GQA 7:1", lambda: W.long_tail_gqa(2)),
]


@pytest.mark.parametrize("name,mk", REFINE_CASES, ids=[c[0] for c in REFINE_CASES])
@pytest.mark.parametrize("num_ctas,c_tile", [(16, 0), (40, 4096), (152, 32768), (3, 0)])
def test_worklist_refinement_bit_exact(oracle_mod, name, mk, num_ctas, c_tile):
    """Move/swap rounds after LPT ("数据并行负载均衡" §4.4 phase 2) on the device
    give the oracle's worklist, and apply as many rounds as the oracle's own
    LPT + refinement of the unit costs."""
    w = mk()
    cu = w.cu_seqlens
    mask = api.mask_for_workload(w)
    dev = torch.device("cuda")
    cu_d = torch.from_numpy(np.ascontiguousarray(cu, dtype=np.int32)).to(dev)
    params = api.make_params(w.num_q_heads, w.num_kv_heads, num_ctas=num_ctas, c_tile=c_tile,
                             refine_iters=20, dispatch=api.DISPATCH_STATIC)
    wl = api.alloc_worklist(cu_d.numel() - 1, mask, params, dev)
    api.build_worklist(cu_d, mask, params, wl)
    torch.cuda.synchronize()
    assert api.worklist_error(wl) == 0
    g = api.decode_worklist(wl)
    om = oracle_mask(w.mask_kind, w.window, w.num_prefix_docs)
    o = oracle_mod.worklist(cu, om, 128, 128, w.num_q_heads, w.num_kv_heads, num_ctas, c_tile,
                            refine_iters=20)
    _assert_same(g, o)
    # rounds: LPT of the enumeration-order costs, then the refinement
    plain = oracle_mod.worklist(cu, om, 128, 128, w.num_q_heads, w.num_kv_heads, num_ctas, c_tile)
    cost = np.zeros(len(plain["units"]), dtype=np.int64)
    cost[plain["units"][:, 0]] = plain["unit_cost"]
    assign, _, _ = oracle_mod.lpt(cost, num_ctas)
    _, _, rounds = oracle_mod.refine_move_swap(cost, assign, num_ctas, 20)
    assert api.worklist_refine_rounds(wl) == rounds


def test_fit_tile_cost_matches_oracle(oracle_mod):
    """The per-tile cost fitted to per-CTA times ("数据并行负载均衡" §4.2), pooled
    over two runs whose worklists were balanced with different per-tile costs:
    the device aggregates and fit equal the oracle's on the same stamps."""
    w = W.long_tail_gqa(2)
    cu = w.cu_seqlens
    dev = torch.device("cuda")
    cu_d = torch.from_numpy(cu).to(dev)
    mask = api.mask_for_workload(w)
    q, k, v = W.workload_qkv(w, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((w.num_q_heads, w.total_tokens), dtype=torch.float32, device=dev)
    nc = torch.cuda.get_device_properties(0).multi_processor_count
    wls, busys, Ps, Us, ts = [], [], [], [], []
    for c_tile in (0, 65536):
        params = api.make_params(w.num_q_heads, w.num_kv_heads, num_ctas=0, c_tile=c_tile,
                                 dispatch=api.DISPATCH_STATIC)
        wl = api.alloc_worklist(w.num_docs, mask, params, dev)
        api.build_worklist(cu_d, mask, params, wl)
        busy = torch.zeros(2 * nc, dtype=torch.int64, device=dev)
        for _ in range(2):
            api.attn_fwd(q, k, v, cu_d, mask, params, wl, out, lse, 0.0, busy)
        torch.cuda.synchronize()
        wls.append(wl)
        busys.append(busy)
        # oracle side: the same worklist from the oracle, the same stamps
        o = oracle_mod.worklist(cu, oracle_mask(w.mask_kind), 128, 128, w.num_q_heads,
                                w.num_kv_heads, nc, c_tile)
        units = o["units"]
        ntiles = np.array([sum(int(r[2] - r[1]) for r in o["runs"][u[7]:u[7] + u[8]])
                           for u in units], dtype=np.int64)
        nsub = np.where(units[:, 5] >= 0, 2, 1)
        P = np.zeros(nc, dtype=np.int64)
        U = np.zeros(nc, dtype=np.int64)
        np.add.at(P, units[:, 9], o["unit_pairs"])
        np.add.at(U, units[:, 9], nsub * (ntiles + 1))
        b = busy.cpu().numpy().reshape(-1, 2)
        has = np.bincount(units[:, 9], minlength=nc) > 0
        Ps.append(P[has])
        Us.append(U[has])
        ts.append((b[has, 1] - b[has, 0]).astype(np.float64))
    ct, coef = api.fit_tile_cost(wls, busys)
    oct_, ocoef = oracle_mod.fit_tile_cost(np.concatenate(Ps), np.concatenate(Us),
                                           np.concatenate(ts))
    assert ct == oct_
    np.testing.assert_allclose(coef, ocoef, rtol=1e-9, atol=1e-12)
    assert 0 <= ct <= 1 << 24 and max(coef) > 0 and min(coef) >= 0


PACK_CASES = [
    ("tiny", lambda: W.tiny_pack(), W.MASK_CAUSAL, 0),
    ("short docs", lambda: W.Workload("short docs", [5, 130, 1, 9, 0, 12, 3, 128, 40, 40, 40,
                                                     8, 15, 127, 1] * 6, 4, 2, 64), W.MASK_CAUSAL, 0),
    ("short docs window", lambda: W.Workload("short docs window", [30, 2, 2, 0, 60, 61, 7, 300, 1]
                                             * 5, 6, 2, 128), W.MASK_SLIDING_WINDOW, 17),
    ("long-tail 2 packs", lambda: W.long_tail_gqa(2), W.MASK_CAUSAL, 0),
]


@pytest.mark.parametrize("name,mk,kind,window", PACK_CASES, ids=[c[0] for c in PACK_CASES])
@pytest.mark.parametrize("dispatch", [api.DISPATCH_STATIC, api.DISPATCH_DYNAMIC])
def test_worklist_packed_short_docs_bit_exact(oracle_mod, name, mk, kind, window, dispatch):
    w = mk()
    cu = w.cu_seqlens
    T = w.total_tokens
    mask = api.make_mask(kind, T, T, window=window)
    g, counts = _gpu_worklist(cu, mask, w.num_q_heads, w.num_kv_heads, 13, 7, dispatch,
                              pack_docs=1)
    o = oracle_mod.worklist(cu, oracle_mask(kind, window), 128, 128, w.num_q_heads,
                            w.num_kv_heads, 13, 7, pack_docs=1)
    assert g["pack_docs"] == 1
    _assert_same(g, o)
    assert counts["pairs_per_head"] == o["pairs_per_head"]
