"""pva_attn_fwd_noalloc: the entry point for callers that cannot allocate
device memory (a plugin in a runtime that owns a fixed memory pool, a
serving process with a memory budget fixed up front, a C host without a
device allocator).  It keeps its worklist in a static device array, so this
test calls it through the C ABI with only inputs and outputs:
- twice in a row on different problems (the array is shared and reused);
  each result must equal pva_build_worklist + pva_attn_fwd with a
  caller-allocated worklist bit for bit (same worklist, same kernel, and the
  dynamic dispatch is deterministic);
- a repeated call leaves the device's free memory unchanged;
- a problem whose worklist is just under the array's size runs, one just
  over it is rejected before any device work;
- cu_seqlens that do not match the mask are reported by pva_noalloc_error.

This file is collected last on purpose; it also passes run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import _lib, api
from packed_varlen_attention_cu_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _reference(q, k, v, cu, mask, params):
    wl = api.alloc_worklist(cu.numel() - 1, mask, params, q.device)
    api.build_worklist(cu, mask, params, wl)
    out = torch.empty((q.shape[0], q.shape[1], q.shape[2]), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    api.attn_fwd(q, k, v, cu, mask, params, wl, out, lse)
    torch.cuda.synchronize()
    assert api.worklist_error(wl) == 0
    return out, lse


def _call(q, k, v, cu, mask, params, out, lse):
    return _lib.lib().pva_attn_fwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), cu.data_ptr(), cu.numel() - 1,
        ctypes.byref(mask), ctypes.byref(params), q.shape[2], out.data_ptr(), 0, lse.data_ptr(),
        0.0, torch.cuda.current_stream().cuda_stream)


def _noalloc_error():
    code = ctypes.c_int32(-1)
    st = _lib.lib().pva_noalloc_error(ctypes.byref(code), torch.cuda.current_stream().cuda_stream)
    assert st == 0, _lib.STATUS_NAMES.get(st, st)
    return int(code.value)


def _outputs(q):
    out = torch.full((q.shape[0], q.shape[1], q.shape[2]), float("nan"), dtype=torch.bfloat16,
                     device=q.device)
    lse = torch.full((q.shape[1], q.shape[0]), float("nan"), dtype=torch.float32, device=q.device)
    return out, lse


def _noalloc(q, k, v, cu, mask, params):
    out, lse = _outputs(q)
    st = _call(q, k, v, cu, mask, params, out, lse)
    assert st == 0, _lib.STATUS_NAMES.get(st, st)
    torch.cuda.synchronize()
    assert _noalloc_error() == 0
    return out, lse


def _problem(w, seed):
    dev = torch.device("cuda")
    q, k, v = W.make_qkv(w.total_tokens, w.total_tokens, w.num_q_heads, w.num_kv_heads,
                         w.head_dim, seed, device="cuda")
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    mask = api.mask_for_workload(w)
    params = api.make_params(w.num_q_heads, w.num_kv_heads, num_ctas=0, c_tile=8192)
    return q.to(dev), k.to(dev), v.to(dev), cu, mask, params


def _equal(got, ref):
    assert torch.equal(got[0], ref[0]), "O differs from the allocating entry point"
    assert torch.equal(got[1], ref[1]), "LSE differs from the allocating entry point"


def test_noalloc_matches_allocating_entry_point_twice():
    problems = [
        _problem(W.tiny_pack(), 1),
        _problem(W.Workload("window GQA", [900, 37, 1300], 8, 2, 128,
                            mask_kind=W.MASK_SLIDING_WINDOW, window=300), 2),
    ]
    for q, k, v, cu, mask, params in problems:  # two calls in a row, different problems
        got = _noalloc(q, k, v, cu, mask, params)
        _equal(got, _reference(q, k, v, cu, mask, params))


def test_noalloc_repeated_call_leaves_free_memory_unchanged():
    q, k, v, cu, mask, params = _problem(W.tiny_pack(), 3)
    out, lse = _outputs(q)
    assert _call(q, k, v, cu, mask, params, out, lse) == 0  # warm-up: module loaded
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        assert _call(q, k, v, cu, mask, params, out, lse) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert _noalloc_error() == 0


def _boundary_tokens(hq, hkv, doc_len, limit):
    """Largest token count of a pack of doc_len-token documents whose worklist
    still fits in `limit` bytes (pva_worklist_bytes is a host computation)."""
    def need(t):
        nd = (t + doc_len - 1) // doc_len
        return api.worklist_bytes(nd, api.make_mask(W.MASK_CAUSAL, t, t),
                                  api.make_params(hq, hkv, num_ctas=0, c_tile=0))
    lo, hi = 1, 1 << 24
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if need(mid) <= limit:
            lo = mid
        else:
            hi = mid
    return lo, need(lo), need(lo + 1)


def test_noalloc_size_limit_at_the_boundary():
    L = _lib.lib()
    limit = L.pva_noalloc_scratch_bytes()
    assert limit == 16 << 20
    hq = hkv = 64
    doc_len, d = 256, 64
    t_in, need_in, need_out = _boundary_tokens(hq, hkv, doc_len, limit)
    assert need_in <= limit < need_out
    # just over: rejected on the host, before any device work (fake pointers)
    t_out = t_in + 1
    nd_out = (t_out + doc_len - 1) // doc_len
    fake = ctypes.c_void_p(256)
    mask_out = api.make_mask(W.MASK_CAUSAL, t_out, t_out)
    params = api.make_params(hq, hkv, num_ctas=0, c_tile=0)
    st = L.pva_attn_fwd_noalloc(fake, fake, fake, fake, nd_out, ctypes.byref(mask_out),
                                ctypes.byref(params), d, fake, 0, fake, 0.0, None)
    assert st == 2  # PVA_ERR_BUFFER_TOO_SMALL
    # just under: runs, equal to the allocating entry point
    lengths = [doc_len] * (t_in // doc_len) + ([t_in % doc_len] if t_in % doc_len else [])
    w = W.Workload("boundary pack", lengths, hq, hkv, d)
    q, k, v, cu, mask, params = _problem(w, 4)
    params.c_tile = 0
    assert api.worklist_bytes(w.num_docs, mask, params) == need_in
    got = _noalloc(q, k, v, cu, mask, params)
    _equal(got, _reference(q, k, v, cu, mask, params))


def test_noalloc_reports_device_errors():
    q, k, v, cu, mask, params = _problem(W.tiny_pack(), 5)
    bad = cu.clone()
    bad[-1] -= 1  # the documents no longer cover the pack's q_tokens rows
    out, lse = _outputs(q)
    assert _call(q, k, v, bad, mask, params, out, lse) == 0  # found on the device
    torch.cuda.synchronize()
    assert _noalloc_error() == 102  # a worklist that does not match the call
    assert torch.isnan(lse).all()  # nothing was written
    # the next good call clears the word
    got = _noalloc(q, k, v, cu, mask, params)
    _equal(got, _reference(q, k, v, cu, mask, params))
