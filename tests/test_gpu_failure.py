"""Failure path of the attention kernel's bounded waits, on the GPU without a
fault: a test hook makes one producer skip one K/V copy (CTA 0's under static
dispatch, that of the CTA which claimed the first LPT rank under dynamic).  The waiting MMA
warps give up after their limit (2 s), the CTA drains its own copies and MMAs,
frees tensor memory and returns; the host reads the wait site from the
worklist's error word, and the same context then runs the pack correctly."""
import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import api, workloads as W

pytestmark = pytest.mark.gpu

TIMEOUT_BASE = 200      # device error code = 200 + wait site
# The MMA warps wait for the withheld item from the start: V_0 (site 5) at
# d = 128; at d = 64, where K_1 is loaded before V_0, K_1 (site 8) or, for a
# single-tile unit, V_0.  The softmax warps' next wait (site 9 or 10) starts
# microseconds later; with up to 200 us between polls either may be the first
# to record its expiry.
SITES = {5, 8, 9, 10}


def _run(w, q, k, v, cu, dispatch):
    m = api.mask_for_workload(w)
    p = api.make_params(w.num_q_heads, w.num_kv_heads, 0, api.default_c_tile(w.head_dim),
                        dispatch=dispatch)
    wl = api.alloc_worklist(w.num_docs, m, p)
    api.build_worklist(cu, m, p, wl)
    out = torch.zeros_like(q)
    lse = torch.zeros((w.num_q_heads, w.total_tokens), dtype=torch.float32, device="cuda")
    busy = torch.zeros(2 * torch.cuda.get_device_properties(0).multi_processor_count,
                       dtype=torch.int64, device="cuda")
    api.attn_fwd(q, k, v, cu, m, p, wl, out, lse, 0.0, busy)
    torch.cuda.synchronize()
    return wl, out, lse, busy


@pytest.mark.parametrize("dispatch", [api.DISPATCH_DYNAMIC, api.DISPATCH_STATIC])
def test_withheld_copy_times_out_and_context_recovers(dispatch):
    w = W.tiny_pack()
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    q, k, v = W.workload_qkv(w, device="cuda")
    wl0, out0, lse0, _ = _run(w, q, k, v, cu, dispatch)
    assert api.worklist_error(wl0) == 0
    try:
        api.debug_withhold_kv_load(True)
        wl1, out1, lse1, busy1 = _run(w, q, k, v, cu, dispatch)
    finally:
        api.debug_withhold_kv_load(False)
    code = api.worklist_error(wl1)
    assert code - TIMEOUT_BASE in SITES, code
    # the CTA gave up after its wait limit (about 2 s), the launch still completed
    b = busy1.cpu().numpy().reshape(-1, 2)
    assert ((b[:, 1] - b[:, 0]) / 1e9).max() > 1.5
    # the context is usable and the next launch is correct again
    wl2, out2, lse2, _ = _run(w, q, k, v, cu, dispatch)
    assert api.worklist_error(wl2) == 0
    assert torch.equal(out2, out0) and torch.equal(lse2, lse0)
