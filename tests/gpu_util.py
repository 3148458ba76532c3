"""Helpers shared by the GPU parity tests: run the library on a problem and
compare with the fp64 oracle at the tolerances of the method's target
(O: max-abs 2e-2 and relative L2 5e-3; LSE: 1e-3 absolute)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from packed_varlen_attention_cu_gb300 import api
from packed_varlen_attention_cu_gb300 import workloads as W

O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
LSE_ABS = 1e-3

ORACLE_MASK_KIND = {W.MASK_CAUSAL: oracle.MASK_CAUSAL,
                    W.MASK_SLIDING_WINDOW: oracle.MASK_SLIDING_WINDOW,
                    W.MASK_SHARED_QUESTION: oracle.MASK_SHARED_QUESTION,
                    W.MASK_ZIGZAG_PAIR: oracle.MASK_ZIGZAG_PAIR,
                    W.MASK_SLICES: oracle.MASK_SLICES,
                    W.MASK_ZIGZAG_STEP: oracle.MASK_ZIGZAG_STEP}


def oracle_mask(kind, window=0, num_prefix=0, cp=0, q_rank=0, k_rank=0, slices=None,
                ring_step=0):
    return oracle.Mask(ORACLE_MASK_KIND[kind], window=window, num_prefix=num_prefix, cp=cp,
                       q_rank=q_rank, k_rank=k_rank, slices=slices, ring_step=ring_step)


def compare(out, lse, ref_o, ref_l, label=""):
    """out/lse: GPU results as float64 numpy; ref: oracle.  Rows with LSE -inf
    must be exactly empty (O = 0, LSE = -inf) on both sides."""
    o = np.asarray(out, dtype=np.float64)
    l = np.asarray(lse, dtype=np.float64)
    assert o.shape == ref_o.shape and l.shape == ref_l.shape, label
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(l), empty), f"{label}: -inf LSE rows differ"
    assert np.isfinite(o).all(), f"{label}: non-finite output"
    err = np.abs(o - ref_o)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref_o))
    rel = float(np.linalg.norm(o - ref_o) / denom) if denom > 0 else max_abs
    fin = ~empty
    lse_err = float(np.abs(l[fin] - ref_l[fin]).max()) if fin.any() else 0.0
    msg = f"{label}: max_abs={max_abs:.3e} rel_l2={rel:.3e} lse_abs={lse_err:.3e}"
    assert max_abs <= O_MAX_ABS, msg
    assert rel <= O_REL_L2, msg
    assert lse_err <= LSE_ABS, msg
    return max_abs, rel, lse_err


def run_gpu(q, k, v, cu_np, mask, hq, hkv, num_ctas=0, c_tile=0, out_fp32=False, scale=0.0,
            dispatch=api.DISPATCH_DYNAMIC, pack_docs=0):
    """Build the worklist and run the forward; returns (out, lse, worklist)."""
    dev = torch.device("cuda")
    cu = torch.from_numpy(np.ascontiguousarray(cu_np, dtype=np.int32)).to(dev)
    params = api.make_params(hq, hkv, num_ctas=num_ctas, c_tile=c_tile, dispatch=dispatch,
                             pack_docs=pack_docs)
    wl = api.alloc_worklist(cu.numel() - 1, mask, params, dev)
    api.build_worklist(cu, mask, params, wl)
    tq, _, d = q.shape
    out = torch.full((tq, hq, d), float("nan"), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                     device=dev)
    lse = torch.full((hq, tq), float("nan"), dtype=torch.float32, device=dev)
    api.attn_fwd(q.to(dev), k.to(dev), v.to(dev), cu, mask, params, wl, out, lse, scale)
    torch.cuda.synchronize()
    err = api.worklist_error(wl)
    assert err == 0, f"device error word {err}"
    return out, lse, wl


def accumulate_gpu(q, k, v, cu_np, mask, hq, hkv, o_run, lse_run, num_ctas=0, c_tile=0,
                   scale=0.0):
    """Build the worklist and run one fused ring step into (o_run, lse_run)."""
    dev = torch.device("cuda")
    cu = torch.from_numpy(np.ascontiguousarray(cu_np, dtype=np.int32)).to(dev)
    params = api.make_params(hq, hkv, num_ctas=num_ctas, c_tile=c_tile)
    wl = api.alloc_worklist(cu.numel() - 1, mask, params, dev)
    api.build_worklist(cu, mask, params, wl)
    api.attn_fwd_accumulate(q.to(dev), k.to(dev), v.to(dev), cu, mask, params, wl, o_run, lse_run,
                            scale)
    torch.cuda.synchronize()
    err = api.worklist_error(wl)
    assert err == 0, f"device error word {err}"
    return wl


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)
