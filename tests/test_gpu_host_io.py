"""pva_attn_fwd_host: the forward pass with inputs and results in host memory
(copies in, worklist, attention, copies out on one stream).  Its results must
be bitwise those of pva_build_worklist + pva_attn_fwd on device buffers, for
pinned and pageable host memory, and with two streams alternating over a few
packs (the way a caller streaming packs overlaps copies with attention)."""
import numpy as np
import pytest
import torch

from packed_varlen_attention_cu_gb300 import api
from packed_varlen_attention_cu_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _device_result(q, k, v, cu_np, mask, params):
    dev = torch.device("cuda")
    cu = torch.from_numpy(cu_np).to(dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    wl = api.alloc_worklist(cu_np.shape[0] - 1, mask, params, dev)
    api.build_worklist(cu, mask, params, wl)
    out = torch.empty_like(qd)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=dev)
    api.attn_fwd(qd, kd, vd, cu, mask, params, wl, out, lse)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def _pack(seed, total, hq, hkv, d):
    lengths = W.lognormal_doc_lengths(total, np.log(700.0), 1.3, 1, total, seed)
    cu_np = W.cu_seqlens_of(lengths)
    T = int(cu_np[-1])
    q, k, v = W.make_qkv(T, T, hq, hkv, d, seed, 1.0)
    return cu_np, q, k, v


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_host_entry_matches_device_path(pinned, d):
    cu_np, q, k, v = _pack(5, 6000, 4, 2, d)
    T = q.shape[0]
    mask = api.make_mask(W.MASK_CAUSAL, T, T)
    params = api.make_params(4, 2, c_tile=api.default_c_tile(d))
    ref_o, ref_l = _device_result(q, k, v, cu_np, mask, params)
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    hq_, hk_, hv_ = pin(q.contiguous()), pin(k.contiguous()), pin(v.contiguous())
    hcu = pin(torch.from_numpy(cu_np))
    o_h = pin(torch.full(q.shape, float("nan"), dtype=torch.bfloat16))
    l_h = pin(torch.full((4, T), float("nan"), dtype=torch.float32))
    bufs = api.alloc_host_path_buffers(hq_, hk_, len(cu_np) - 1, mask, params)
    api.attn_fwd_host(hq_, hk_, hv_, hcu, len(cu_np) - 1, mask, params, o_h, l_h, bufs)
    torch.cuda.synchronize()
    assert api.worklist_error(bufs["worklist"]) == 0
    assert torch.equal(o_h, ref_o) and torch.equal(l_h, ref_l)


def test_two_streams_alternating_over_packs():
    d, hq, hkv = 128, 4, 2
    packs = [_pack(s, 5000, hq, hkv, d) for s in range(4)]
    T = min(p[1].shape[0] for p in packs)
    assert all(p[1].shape[0] == T for p in packs)  # every pack fills its total
    streams = [torch.cuda.Stream() for _ in range(2)]
    mask = api.make_mask(W.MASK_CAUSAL, T, T)
    params = api.make_params(hq, hkv, c_tile=api.default_c_tile(d))
    host = []
    for cu_np, q, k, v in packs:
        host.append({"q": q.contiguous().pin_memory(), "k": k.contiguous().pin_memory(),
                     "v": v.contiguous().pin_memory(), "cu": torch.from_numpy(cu_np).pin_memory(),
                     "o": torch.empty(q.shape, dtype=torch.bfloat16).pin_memory(),
                     "l": torch.empty((hq, T), dtype=torch.float32).pin_memory(),
                     "nd": len(cu_np) - 1})
    # buffers are sized for the largest document count among the packs
    nd_max = max(h["nd"] for h in host)
    bufs = [api.alloc_host_path_buffers(host[0]["q"], host[0]["k"], nd_max, mask, params)
            for _ in range(2)]
    for i, h in enumerate(host):
        api.attn_fwd_host(h["q"], h["k"], h["v"], h["cu"], h["nd"], mask, params, h["o"], h["l"],
                          bufs[i % 2], 0.0, streams[i % 2])
    torch.cuda.synchronize()
    for b in bufs:
        assert api.worklist_error(b["worklist"]) == 0
    for (cu_np, q, k, v), h in zip(packs, host):
        ref_o, ref_l = _device_result(q, k, v, cu_np, mask, params)
        assert torch.equal(h["o"], ref_o) and torch.equal(h["l"], ref_l)
