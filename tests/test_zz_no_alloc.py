"""pva_attn_fwd_noalloc: the entry point for callers that cannot allocate
device memory (a plugin in a runtime that owns a fixed memory pool, a
serving process with a memory budget fixed up front, a C host without a
device allocator).  It keeps its worklist in a static device array, so this
test calls it through the C ABI with only inputs and outputs, twice in a row
on different problems (the array is shared and reused), and checks each
result against pva_build_worklist + pva_attn_fwd with a caller-allocated
worklist, within the tolerances of the other attention tests.

This file is collected last on purpose; it also passes run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import _lib, api
from packed_varlen_attention_cu_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_REL_L2, LSE_ABS = 2e-2, 5e-3, 1e-3


def _reference(q, k, v, cu, mask, params):
    wl = api.alloc_worklist(cu.numel() - 1, mask, params, q.device)
    api.build_worklist(cu, mask, params, wl)
    out = torch.empty((q.shape[0], q.shape[1], q.shape[2]), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    api.attn_fwd(q, k, v, cu, mask, params, wl, out, lse)
    return out, lse


def _noalloc(q, k, v, cu, mask, params):
    out = torch.full((q.shape[0], q.shape[1], q.shape[2]), float("nan"), dtype=torch.bfloat16,
                     device=q.device)
    lse = torch.full((q.shape[1], q.shape[0]), float("nan"), dtype=torch.float32, device=q.device)
    st = _lib.lib().pva_attn_fwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), cu.data_ptr(), cu.numel() - 1,
        ctypes.byref(mask), ctypes.byref(params), q.shape[2], out.data_ptr(), 0, lse.data_ptr(),
        0.0, torch.cuda.current_stream().cuda_stream)
    assert st == 0, _lib.STATUS_NAMES.get(st, st)
    return out, lse


def _close(a, b):
    a_o, a_l = a[0].double(), a[1].double()
    b_o, b_l = b[0].double(), b[1].double()
    assert torch.isfinite(a_o).all() and torch.isfinite(a_l).all()
    assert (a_o - b_o).abs().max().item() <= O_MAX_ABS
    assert ((a_o - b_o).norm() / b_o.norm()).item() <= O_REL_L2
    assert (a_l - b_l).abs().max().item() <= LSE_ABS


def _problem(w, seed):
    dev = torch.device("cuda")
    q, k, v = W.make_qkv(w.total_tokens, w.total_tokens, w.num_q_heads, w.num_kv_heads,
                         w.head_dim, seed)
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    mask = api.mask_for_workload(w)
    params = api.make_params(w.num_q_heads, w.num_kv_heads, num_ctas=0, c_tile=8192)
    return q.to(dev), k.to(dev), v.to(dev), cu, mask, params


def test_noalloc_matches_allocating_entry_point_twice():
    problems = [
        _problem(W.tiny_pack(), 1),
        _problem(W.Workload("window GQA", [900, 37, 1300], 8, 2, 128,
                            mask_kind=W.MASK_SLIDING_WINDOW, window=300), 2),
    ]
    for q, k, v, cu, mask, params in problems:  # two calls in a row, different problems
        got = _noalloc(q, k, v, cu, mask, params)
        torch.cuda.synchronize()
        ref = _reference(q, k, v, cu, mask, params)
        torch.cuda.synchronize()
        _close(got, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = _lib.lib()
    assert L.pva_noalloc_scratch_bytes() == 16 << 20
    # a 4M-token pack with 32 q heads needs more worklist than the static array holds
    mask = api.make_mask(W.MASK_CAUSAL, 1 << 22, 1 << 22)
    params = api.make_params(32, 8, num_ctas=0, c_tile=0)
    assert api.worklist_bytes(64, mask, params) > L.pva_noalloc_scratch_bytes()
    fake = ctypes.c_void_p(256)
    st = L.pva_attn_fwd_noalloc(fake, fake, fake, fake, 64, ctypes.byref(mask),
                                ctypes.byref(params), 128, fake, 0, fake, 0.0, None)
    assert st == 2  # PVA_ERR_BUFFER_TOO_SMALL, before any device work
