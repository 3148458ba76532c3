"""tcgen05 attention forward vs the fp64 oracle.

Small packs are compared element by element on every row and head; the full
workloads (128K pack, Libra pair, long-tail GQA batch, shared question,
sliding window) on sampled rows that the oracle computes one by one, in the
same launch configuration the benchmark times (one CTA per SM).
Tolerances: O max-abs 2e-2 and relative L2 5e-3, LSE 1e-3 absolute.
"""
import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import api
from packed_varlen_attention_cu_gb300 import workloads as W

from gpu_util import compare, oracle_mask, run_gpu, to_np

pytestmark = pytest.mark.gpu


def _full_check(oracle_mod, lengths, hq, hkv, d, kind=W.MASK_CAUSAL, window=0, num_prefix=0,
                seed=0, out_fp32=False, num_ctas=0, c_tile=0, scale_v=1.0,
                dispatch=api.DISPATCH_DYNAMIC):
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, T, hq, hkv, d, seed, scale_v)
    mask = api.make_mask(kind, T, T, window=window, num_prefix_docs=num_prefix)
    out, lse, _ = run_gpu(q, k, v, cu, mask, hq, hkv, num_ctas=num_ctas, c_tile=c_tile,
                          out_fp32=out_fp32, dispatch=dispatch)
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu,
                                        oracle_mask(kind, window, num_prefix))
    return compare(to_np(out), to_np(lse), ref_o, ref_l, f"{lengths[:4]} h{hq}/{hkv} d{d}")


def test_tiny_pack_config(oracle_mod):
    w = W.tiny_pack()
    _full_check(oracle_mod, w.lengths, 4, 4, 64)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(1, 1), (2, 2), (4, 1), (6, 2), (7, 1)])
def test_causal_docs_heads(oracle_mod, d, hq, hkv):
    # several tiles per document and ragged tails: 1..3 q tiles, partial kv tiles
    lengths = [300, 1, 128, 129, 0, 17, 256, 413]
    _full_check(oracle_mod, lengths, hq, hkv, d, seed=hq * 10 + d)


@pytest.mark.parametrize("d", [64, 128])
def test_fp32_partial_output(oracle_mod, d):
    _full_check(oracle_mod, [700, 33, 260], 4, 2, d, out_fp32=True, seed=5)


@pytest.mark.parametrize("window", [1, 5, 128, 200, 1000])
def test_sliding_window(oracle_mod, window):
    _full_check(oracle_mod, [1100, 64, 400], 4, 2, 128, kind=W.MASK_SLIDING_WINDOW,
                window=window, seed=window)


@pytest.mark.parametrize("num_prefix", [1, 2])
def test_shared_question(oracle_mod, num_prefix):
    _full_check(oracle_mod, [500, 130, 300, 256, 77], 4, 1, 128, kind=W.MASK_SHARED_QUESTION,
                num_prefix=num_prefix, seed=num_prefix)


@pytest.mark.parametrize("d", [64, 128])
def test_single_long_document_many_tiles(oracle_mod, d):
    _full_check(oracle_mod, [3000], 2, 1, d, seed=9, scale_v=0.5)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dispatch", [api.DISPATCH_DYNAMIC, api.DISPATCH_STATIC])
def test_zero_length_and_single_token_documents(oracle_mod, d, dispatch):
    """Degenerate packs: empty documents between others, one-token documents,
    and far fewer units than CTAs (most CTAs claim nothing but the end)."""
    _full_check(oracle_mod, [0, 1, 0, 5, 0, 0, 130, 1, 0], 4, 2, d, seed=17, dispatch=dispatch)
    _full_check(oracle_mod, [1] * 37, 2, 1, d, seed=18, dispatch=dispatch)


def test_d64_odd_group_and_single_tile_units(oracle_mod):
    """d = 64 with an odd GQA group (its last head pairs consecutive q tiles, so
    some units have one sub-tile) and documents of one tile or less: the split-P
    pipeline's K_{j+1}-before-V_j order with one-tile units and idle issuers."""
    _full_check(oracle_mod, [100, 128, 129, 40, 700, 1, 255, 900], 7, 1, 64, seed=13)


@pytest.mark.parametrize("dispatch", [api.DISPATCH_DYNAMIC, api.DISPATCH_STATIC])
@pytest.mark.parametrize("num_ctas,c_tile", [(1, 0), (3, 100), (1024, 0)])
def test_cta_counts(oracle_mod, num_ctas, c_tile, dispatch):
    _full_check(oracle_mod, [520, 130, 900], 4, 2, 64, num_ctas=num_ctas, c_tile=c_tile, seed=4,
                dispatch=dispatch)


@pytest.mark.parametrize("d", [64, 128])
def test_dynamic_and_static_dispatch_agree_bitwise(d):
    """A unit computes the same bits whichever CTA runs it: dynamic dispatch
    (units claimed in LPT order at run time) and the static per-CTA lists give
    identical outputs, and repeated launches on one worklist (whose claim
    counter the last CTA resets) repeat them."""
    lengths = [int(x) for x in W.lognormal_doc_lengths(12000, np.log(900.0), 1.2, 1, 6000, 3)]
    cu_np = W.cu_seqlens_of(lengths)
    T = int(cu_np[-1])
    q, k, v = (x.cuda() for x in W.make_qkv(T, T, 4, 2, d, 11, 1.0))
    mask = api.make_mask(W.MASK_CAUSAL, T, T)
    cu = torch.from_numpy(cu_np).cuda()
    res = {}
    for disp in (api.DISPATCH_STATIC, api.DISPATCH_DYNAMIC):
        params = api.make_params(4, 2, c_tile=api.default_c_tile(d), dispatch=disp)
        wl = api.alloc_worklist(len(lengths), mask, params)
        api.build_worklist(cu, mask, params, wl)
        runs = []
        for _ in range(3):
            out = torch.empty_like(q)
            lse = torch.empty((4, T), dtype=torch.float32, device="cuda")
            api.attn_fwd(q, k, v, cu, mask, params, wl, out, lse, 0.0)
            runs.append((out, lse))
        torch.cuda.synchronize()
        assert api.worklist_error(wl) == 0
        for o, l in runs[1:]:
            assert torch.equal(o, runs[0][0]) and torch.equal(l, runs[0][1])
        res[disp] = runs[0]
    assert torch.equal(res[api.DISPATCH_STATIC][0], res[api.DISPATCH_DYNAMIC][0])
    assert torch.equal(res[api.DISPATCH_STATIC][1], res[api.DISPATCH_DYNAMIC][1])


@pytest.mark.parametrize("d", [64, 128])
def test_large_logits_rescale_path(oracle_mod, d):
    # scaled inputs push the running max up across kv tiles (exercises O rescaling;
    # at d = 64 after the wait for the previous tile's PV, P being apart from S)
    lengths = [1500, 700]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, T, 2, 2, d, 21)
    ramp = torch.linspace(0.2, 3.0, T).to(torch.bfloat16)[:, None, None]
    k = (k.float() * ramp.float()).to(torch.bfloat16)
    q = (q.float() * 2.0).to(torch.bfloat16)
    mask = api.make_mask(W.MASK_CAUSAL, T, T)
    out, lse, _ = run_gpu(q, k, v, cu, mask, 2, 2)
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu, oracle_mask(W.MASK_CAUSAL))
    compare(to_np(out), to_np(lse), ref_o, ref_l, "rescale")


def test_explicit_slices_and_unwritten_rows(oracle_mod):
    T = 705
    sl = np.array([[0, 300, 0, 0, 300, 0, 1, 0],
                   [300, 200, 1000, 0, 150, 0, 0, 0],
                   [300, 200, 1000, 300, 400, 900, 1, 64],
                   [700, 5, 0, 700, 5, 0, 1, 0]], dtype=np.int32)
    q, k, v = W.make_qkv(T, T, 2, 1, 64, 6)
    mask = api.make_mask(W.MASK_SLICES, T, T, slices=sl)
    out, lse, _ = run_gpu(q, k, v, np.array([0, T], dtype=np.int32), mask, 2, 1, out_fp32=True)
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), np.array([0, T], dtype=np.int32),
                                        oracle_mask(W.MASK_SLICES, slices=sl))
    rows = np.r_[0:500, 700:705]
    compare(to_np(out)[rows], to_np(lse)[:, rows], ref_o[rows], ref_l[:, rows], "slices")
    # rows outside every slice are left untouched
    assert torch.isnan(out[500:700]).all() and torch.isnan(lse[:, 500:700]).all()


@pytest.mark.parametrize("d", [64, 128])
def test_inv_and_bi_causal_slices(oracle_mod, d):
    # INV-CAUSAL (with and without a window), BI-CAUSAL on a 200 x 300 rectangle,
    # CAUSAL with a window and FULL, over three query segments; ragged tiles
    sl = np.array([[0, 300, 0, 0, 300, 0, 2, 0],
                   [300, 200, 1000, 300, 300, 1000, 3, 0],
                   [300, 200, 1000, 0, 300, 900, 1, 64],
                   [500, 400, 0, 600, 300, 50, 2, 200],
                   [500, 400, 0, 300, 300, 0, 0, 0]], dtype=np.int32)
    T = 900
    q, k, v = W.make_qkv(T, T, 4, 2, d, 40 + d)
    mask = api.make_mask(W.MASK_SLICES, T, T, slices=sl)
    out, lse, _ = run_gpu(q, k, v, np.array([0, T], dtype=np.int32), mask, 4, 2)
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(q), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), np.array([0, T], dtype=np.int32),
                                        oracle_mask(W.MASK_SLICES, slices=sl))
    compare(to_np(out), to_np(lse), ref_o, ref_l, f"inv/bi slices d{d}")


@pytest.mark.parametrize("cp", [2, 4])
def test_zigzag_pairs_each_partial(oracle_mod, cp):
    lengths = [700, 3, 260, 1100, 40]
    cu = W.cu_seqlens_of(lengths)
    T = int(cu[-1])
    q, k, v = W.make_qkv(T, T, 4, 2, 128, 12)
    maps = [oracle_mod.zigzag_map(cu, cp, r)[0] for r in range(cp)]
    for r in range(cp):
        for s in range(cp):
            mask = api.make_mask(W.MASK_ZIGZAG_PAIR, len(maps[r]), len(maps[s]), cp=cp, q_rank=r,
                                 k_rank=s)
            qr, ks, vs = q[maps[r]], k[maps[s]], v[maps[s]]
            out, lse, _ = run_gpu(qr, ks, vs, cu, mask, 4, 2, out_fp32=True)
            ref_o, ref_l = oracle_mod.attention(
                oracle_mod.bf16_bits(qr), oracle_mod.bf16_bits(ks), oracle_mod.bf16_bits(vs), cu,
                oracle_mask(W.MASK_ZIGZAG_PAIR, cp=cp, q_rank=r, k_rank=s))
            compare(to_np(out), to_np(lse), ref_o, ref_l, f"zigzag r{r} s{s}")


# ----------------------------------------------------------------- full sizes
FULL = [
    ("128K causal pack", W.zigzag_pack),
    ("libra pair", W.libra_pair),
    ("long-tail GQA 8 packs", W.long_tail_gqa),
    ("shared question", W.shared_question),
    ("sliding window", W.sliding_window),
]


@pytest.mark.parametrize("name,mk", FULL, ids=[f[0] for f in FULL])
def test_full_size_sampled_rows(oracle_mod, name, mk):
    w = mk()
    dev = torch.device("cuda")
    cu = w.cu_seqlens
    T = w.total_tokens
    q, k, v = W.workload_qkv(w, device="cuda")
    mask = api.mask_for_workload(w)
    out, lse, _ = run_gpu(q, k, v, cu, mask, w.num_q_heads, w.num_kv_heads)
    # sample: random rows + every document's first, last and 128-boundary rows
    special = []
    for a, b in zip(cu[:-1], cu[1:]):
        if b > a:
            special += [a, b - 1, min(a + 127, b - 1), min(a + 128, b - 1)]
    jobs = W.random_rows(T, w.num_q_heads, 192, seed=17, must_include=special)
    jt = torch.from_numpy(jobs).long()
    qs = q[jt[:, 0].to(dev)].cpu()  # rows of the sampled jobs
    # the oracle takes the full K/V and only the sampled query rows
    qfull = torch.zeros((T, w.num_q_heads, w.head_dim), dtype=torch.bfloat16)
    qfull[jt[:, 0]] = qs
    ref_o, ref_l = oracle_mod.attention(oracle_mod.bf16_bits(qfull), oracle_mod.bf16_bits(k),
                                        oracle_mod.bf16_bits(v), cu,
                                        oracle_mask(w.mask_kind, w.window, w.num_prefix_docs),
                                        jobs=jobs)
    got_o = to_np(out[jt[:, 0].to(dev), jt[:, 1].to(dev)])
    got_l = to_np(lse[jt[:, 1].to(dev), jt[:, 0].to(dev)])
    compare(got_o, got_l, ref_o, ref_l, name)
    # properties that hold on every row: finite output, finite LSE (each row sees itself)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
