"""Thin Python binding of the C ABI (include/pva.h).

Argument marshalling only: tensors are passed by ``data_ptr()`` and the
current CUDA stream; every step of the computation runs in the library's
kernels.  PyTorch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np
import torch

from . import _lib
from ._lib import MaskDesc, Slice, WorklistParams, check, lib
from .workloads import (MASK_CAUSAL, MASK_SHARED_QUESTION, MASK_SLICES, MASK_SLIDING_WINDOW,
                        MASK_ZIGZAG_PAIR, MASK_ZIGZAG_STEP)

SLICE_FULL, SLICE_CAUSAL, SLICE_INV_CAUSAL, SLICE_BI_CAUSAL = 0, 1, 2, 3
TILE = 128


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def make_mask(kind: int = MASK_CAUSAL, q_tokens: int = 0, k_tokens: int = 0, window: int = 0,
              num_prefix_docs: int = 0, cp: int = 0, q_rank: int = 0, k_rank: int = 0,
              slices: Optional[np.ndarray] = None, ring_step: int = 0) -> MaskDesc:
    """pva_mask_desc.  ``slices``: int32 [n, 8] rows (q_row0, q_len, q_pos0, k_row0, k_len,
    k_pos0, type, window); the array is kept alive on the returned object."""
    m = MaskDesc()
    m.kind, m.window, m.num_prefix_docs = kind, window, num_prefix_docs
    m.cp, m.q_rank, m.k_rank = cp, q_rank, k_rank
    m.ring_step = ring_step
    m.q_tokens, m.k_tokens = q_tokens, k_tokens
    if slices is not None:
        arr = np.ascontiguousarray(slices, dtype=np.int32).reshape(-1, 8)
        m._slices_keep = arr
        m.slices = arr.ctypes.data_as(ctypes.POINTER(Slice))
        m.num_slices = arr.shape[0]
    return m


DISPATCH_DYNAMIC, DISPATCH_STATIC = 0, 1  # pva_dispatch

# Kernels one pva_build_worklist launches: plan, units, then for static
# dispatch chunk sort + merge rank (LPT order), LPT, chunk sort + merge rank
# (per-CTA order); for dynamic dispatch chunk sort + merge rank (dispatch order).
def worklist_build_kernels(params) -> int:
    return 4 if params.dispatch == DISPATCH_DYNAMIC else 7


def default_c_tile(head_dim: int) -> int:
    """Per-tile fixed cost (pair units) that balanced CTA busy time best on GB300:
    a computed 128 x 128 tile costs about its 16384 pairs of MMA work plus a
    softmax/hand-off term that does not shrink with the head dimension, so the
    fixed term doubles when d halves (32768 at d = 128, 65536 at d = 64)."""
    return 32768 * 128 // int(head_dim)


def make_params(num_q_heads: int, num_kv_heads: int, num_ctas: int = 0, c_tile: int = 0,
                tile_m: int = TILE, tile_n: int = TILE, refine_iters: int = 0,
                dispatch: int = DISPATCH_DYNAMIC, pack_docs: int = 0) -> WorklistParams:
    """pva_worklist_params.  pack_docs = 1: short documents share tiles."""
    p = WorklistParams()
    p.refine_iters = refine_iters
    p.dispatch = dispatch
    p.pack_docs = pack_docs
    p.tile_m, p.tile_n = tile_m, tile_n
    p.num_q_heads, p.num_kv_heads = num_q_heads, num_kv_heads
    p.num_ctas, p.c_tile = num_ctas, c_tile
    return p


def worklist_bytes(num_docs: int, mask: MaskDesc, params: WorklistParams) -> int:
    n = lib().pva_worklist_bytes(num_docs, ctypes.byref(mask), ctypes.byref(params))
    if n == 0:
        raise _lib.PvaError("pva_worklist_bytes", 1)
    return int(n)


def alloc_worklist(num_docs: int, mask: MaskDesc, params: WorklistParams,
                   device="cuda") -> torch.Tensor:
    """Caller-owned device buffer for the worklist (256-byte aligned by the allocator)."""
    return torch.empty(worklist_bytes(num_docs, mask, params), dtype=torch.uint8, device=device)


def build_worklist(cu_seqlens: Optional[torch.Tensor], mask: MaskDesc, params: WorklistParams,
                   worklist: torch.Tensor, stream=None) -> None:
    nd = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None:
        assert cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda
    check("pva_build_worklist", lib().pva_build_worklist(
        _ptr(cu_seqlens), nd, ctypes.byref(mask), ctypes.byref(params), _ptr(worklist),
        worklist.numel(), _stream(stream)))


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
             cu_seqlens: Optional[torch.Tensor], mask: MaskDesc, params: WorklistParams,
             worklist: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
             softmax_scale: float = 0.0, cta_busy: Optional[torch.Tensor] = None,
             stream=None) -> None:
    """out [Tq, Hq, d] bf16 or fp32, lse [Hq, Tq] fp32 (written by the kernel)."""
    for t in (q, k, v, out, lse):
        assert t.is_cuda and t.is_contiguous()
    assert q.dtype == k.dtype == v.dtype == torch.bfloat16
    assert lse.dtype == torch.float32 and out.dtype in (torch.bfloat16, torch.float32)
    check("pva_attn_fwd", lib().pva_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), ctypes.byref(mask), ctypes.byref(params),
        q.shape[-1], _ptr(worklist), _ptr(out), 1 if out.dtype == torch.float32 else 0,
        _ptr(lse), float(softmax_scale), _ptr(cta_busy), _stream(stream)))


def attn_fwd_host(q_host: torch.Tensor, k_host: torch.Tensor, v_host: torch.Tensor,
                  cu_host: Optional[torch.Tensor], num_docs: int, mask: MaskDesc,
                  params: WorklistParams, out_host: torch.Tensor, lse_host: torch.Tensor,
                  dev_bufs: dict, softmax_scale: float = 0.0, stream=None) -> None:
    """pva_attn_fwd_host: copies in, worklist, attention and copies out on one
    stream.  Host tensors (pinned for asynchronous copies) hold the inputs and
    receive O and LSE; dev_bufs holds the device buffers "q", "k", "v", "cu",
    "worklist", "out", "lse" (see alloc_host_path_buffers)."""
    for t in (q_host, k_host, v_host, out_host, lse_host):
        assert not t.is_cuda and t.is_contiguous()
    wl = dev_bufs["worklist"]
    check("pva_attn_fwd_host", lib().pva_attn_fwd_host(
        _ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(cu_host), num_docs, ctypes.byref(mask),
        ctypes.byref(params), q_host.shape[-1], _ptr(out_host), _ptr(lse_host),
        float(softmax_scale), _ptr(dev_bufs["q"]), _ptr(dev_bufs["k"]), _ptr(dev_bufs["v"]),
        _ptr(dev_bufs["cu"]), _ptr(wl), wl.numel(), _ptr(dev_bufs["out"]), _ptr(dev_bufs["lse"]),
        _stream(stream)))


def alloc_host_path_buffers(q_host: torch.Tensor, k_host: torch.Tensor, num_docs: int,
                            mask: MaskDesc, params: WorklistParams, device=None) -> dict:
    """Device buffers for attn_fwd_host with the shapes of q_host / k_host."""
    dev = device or torch.device("cuda")
    tq, hq, d = q_host.shape
    return {"q": torch.empty(q_host.shape, dtype=torch.bfloat16, device=dev),
            "k": torch.empty(k_host.shape, dtype=torch.bfloat16, device=dev),
            "v": torch.empty(k_host.shape, dtype=torch.bfloat16, device=dev),
            "cu": torch.empty((num_docs + 1,), dtype=torch.int32, device=dev),
            "worklist": alloc_worklist(num_docs, mask, params, dev),
            "out": torch.empty((tq, hq, d), dtype=torch.bfloat16, device=dev),
            "lse": torch.empty((hq, tq), dtype=torch.float32, device=dev)}


def attn_fwd_accumulate(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        cu_seqlens: Optional[torch.Tensor], mask: MaskDesc,
                        params: WorklistParams, worklist: torch.Tensor, o_run: torch.Tensor,
                        lse_run: torch.Tensor, softmax_scale: float = 0.0,
                        cta_busy: Optional[torch.Tensor] = None, stream=None) -> None:
    """Fused ring step: merge this call's attention into the running fp32
    o_run [Tq, Hq, d] and lse_run [Hq, Tq] in place (start with lse_run = -inf)."""
    for t in (q, k, v, o_run, lse_run):
        assert t.is_cuda and t.is_contiguous()
    assert q.dtype == k.dtype == v.dtype == torch.bfloat16
    assert o_run.dtype == lse_run.dtype == torch.float32
    check("pva_attn_fwd_accumulate", lib().pva_attn_fwd_accumulate(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), ctypes.byref(mask), ctypes.byref(params),
        q.shape[-1], _ptr(worklist), _ptr(o_run), _ptr(lse_run), float(softmax_scale),
        _ptr(cta_busy), _stream(stream)))


def zigzag_shard_len(cu_seqlens_host: np.ndarray, cp: int, rank: int) -> int:
    cu = np.ascontiguousarray(cu_seqlens_host, dtype=np.int32)
    n = lib().pva_zigzag_shard_len(cu.ctypes.data_as(ctypes.c_void_p), cu.shape[0] - 1, cp, rank)
    if n < 0:
        raise _lib.PvaError("pva_zigzag_shard_len", 1)
    return int(n)


def zigzag_shard(cu_seqlens: torch.Tensor, cp: int, rank: int, gather_map: torch.Tensor,
                 chunk_table: Optional[torch.Tensor] = None, stream=None) -> None:
    check("pva_zigzag_shard", lib().pva_zigzag_shard(
        _ptr(cu_seqlens), cu_seqlens.numel() - 1, cp, rank, _ptr(gather_map), _ptr(chunk_table),
        _stream(stream)))


def zigzag_ring_map(cu_seqlens: torch.Tensor, cp: int, ring_map: torch.Tensor,
                    stream=None) -> None:
    """Ring order of all cp zigzag shards (pva_zigzag_ring_map) into ring_map [T] int32."""
    check("pva_zigzag_ring_map", lib().pva_zigzag_ring_map(
        _ptr(cu_seqlens), cu_seqlens.numel() - 1, cp, _ptr(ring_map), _stream(stream)))


def gather_rows(src: torch.Tensor, index_map: torch.Tensor, dst: torch.Tensor,
                scatter: bool = False, stream=None) -> None:
    """dst[i] = src[map[i]] (or dst[map[i]] = src[i]) over the first dimension."""
    rows = index_map.numel()
    # the library sees raw pointers: the map's own side must hold `rows` rows
    if (src if scatter else dst).shape[0] < rows:
        raise ValueError("gather_rows: the map has more entries than the tensor it fills has rows")
    row_bytes = src[0].numel() * src.element_size()
    indexed = dst.shape[0] if scatter else src.shape[0]
    check("pva_gather_rows", lib().pva_gather_rows(
        _ptr(src), _ptr(index_map), _ptr(dst), rows, row_bytes, indexed, 1 if scatter else 0,
        _stream(stream)))


def merge_partials(o_a: torch.Tensor, lse_a: torch.Tensor, o_b: torch.Tensor,
                   lse_b: torch.Tensor, out: torch.Tensor, lse_out: torch.Tensor,
                   stream=None) -> None:
    tokens, heads, d = o_a.shape
    check("pva_merge_partials", lib().pva_merge_partials(
        _ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(out), _ptr(lse_out), tokens, heads,
        d, 1 if o_a.dtype == torch.float32 else 0, _stream(stream)))


def worklist_error(worklist: torch.Tensor, stream=None) -> int:
    code = ctypes.c_int32(0)
    check("pva_worklist_error", lib().pva_worklist_error(_ptr(worklist), ctypes.byref(code),
                                                         _stream(stream)))
    return int(code.value)


def fit_tile_cost(worklists: Sequence[torch.Tensor], cta_busy: Sequence[torch.Tensor],
                  stream=None):
    """Per-tile cost fitted to the per-CTA times of several runs (one worklist and
    one busy-stamp tensor per run): (c_tile, (a ns per pair, c ns per tile))."""
    n = len(worklists)
    assert n == len(cta_busy) and n > 0
    wl = (ctypes.c_void_p * n)(*[w.data_ptr() for w in worklists])
    bz = (ctypes.c_void_p * n)(*[b.data_ptr() for b in cta_busy])
    ct = ctypes.c_int64(0)
    coef = (ctypes.c_double * 2)()
    check("pva_fit_tile_cost", lib().pva_fit_tile_cost(wl, bz, n, ctypes.byref(ct), coef,
                                                       _stream(stream)))
    return int(ct.value), (coef[0], coef[1])


def worklist_refine_rounds(worklist: torch.Tensor) -> int:
    """Move/swap rounds the worklist build applied after LPT (header field)."""
    off = _HDR.itemsize + 8  # after lpt_steps and refine_iters
    return int(np.frombuffer(worklist[off:off + 4].cpu().numpy().tobytes(), dtype="<i4")[0])


# ------------------------------------------------------ backward
def bwd_plan_bytes(num_docs: int, mask: MaskDesc, params: WorklistParams) -> int:
    n = lib().pva_bwd_plan_bytes(num_docs, ctypes.byref(mask), ctypes.byref(params))
    if n == 0:
        raise _lib.PvaError("pva_bwd_plan_bytes", 4)
    return int(n)


def alloc_bwd_plan(num_docs: int, mask: MaskDesc, params: WorklistParams,
                   device="cuda") -> torch.Tensor:
    return torch.empty(bwd_plan_bytes(num_docs, mask, params), dtype=torch.uint8, device=device)


def build_bwd_plan(worklist: torch.Tensor, num_docs: int, mask: MaskDesc,
                   params: WorklistParams, plan: torch.Tensor, stream=None) -> None:
    check("pva_build_bwd_plan", lib().pva_build_bwd_plan(
        _ptr(worklist), num_docs, ctypes.byref(mask), ctypes.byref(params), _ptr(plan),
        plan.numel(), _stream(stream)))


def attn_bwd(q, k, v, out, lse, dout, cu_seqlens: Optional[torch.Tensor], num_docs: int,
             mask: MaskDesc, params: WorklistParams, worklist: torch.Tensor, plan: torch.Tensor,
             dq: torch.Tensor, dk: torch.Tensor, dv: torch.Tensor, softmax_scale: float = 0.0,
             stream=None) -> None:
    """Gradients into dq [Tq, Hq, d], dk/dv [Tk, Hkv, d] (all bf16 or all fp32)."""
    for t in (q, k, v, out, lse, dout, dq, dk, dv):
        assert t.is_cuda and t.is_contiguous()
    assert dq.dtype == dk.dtype == dv.dtype and dq.dtype in (torch.bfloat16, torch.float32)
    check("pva_attn_bwd", lib().pva_attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(cu_seqlens), num_docs,
        ctypes.byref(mask), ctypes.byref(params), q.shape[-1], _ptr(worklist), _ptr(plan),
        _ptr(dq), _ptr(dk), _ptr(dv), 1 if dq.dtype == torch.float32 else 0,
        float(softmax_scale), _stream(stream)))


# ------------------------------------------------------ sharding solvers
def chunk_areas(cu_seqlens: torch.Tensor, mask: MaskDesc, chunk_size: int,
                areas: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Allowed pairs of every chunk of chunk_size query rows (device int64)."""
    n = (mask.q_tokens + chunk_size - 1) // chunk_size
    if areas is None:
        areas = torch.empty((n,), dtype=torch.int64, device=cu_seqlens.device)
    check("pva_chunk_areas", lib().pva_chunk_areas(
        _ptr(cu_seqlens), cu_seqlens.numel() - 1, ctypes.byref(mask), chunk_size, _ptr(areas),
        _stream(stream)))
    return areas


def dispatch_chunks(areas: torch.Tensor, cp: int, bucket: Optional[torch.Tensor] = None,
                    bucket_area: Optional[torch.Tensor] = None, stream=None):
    """Greedy min-heap dispatch: (bucket [n] int32, bucket_area [cp] int64), device."""
    n = areas.numel()
    if bucket is None:
        bucket = torch.empty((max(n, 1),), dtype=torch.int32, device=areas.device)
    if bucket_area is None:
        bucket_area = torch.empty((cp,), dtype=torch.int64, device=areas.device)
    check("pva_dispatch_chunks", lib().pva_dispatch_chunks(
        _ptr(areas), n, cp, _ptr(bucket), _ptr(bucket_area), _stream(stream)))
    return bucket[:n], bucket_area


def striped_shard_len(total_tokens: int, cp: int, rank: int, stripe: int) -> int:
    n = lib().pva_striped_shard_len(total_tokens, cp, rank, stripe)
    if n < 0:
        raise _lib.PvaError("pva_striped_shard_len", 1)
    return int(n)


def striped_shard(total_tokens: int, cp: int, rank: int, stripe: int, map_out: torch.Tensor,
                  stream=None) -> None:
    check("pva_striped_shard", lib().pva_striped_shard(
        total_tokens, cp, rank, stripe, _ptr(map_out), _stream(stream)))


def wlb_choose(cu_seqlens_host: np.ndarray, cp: int, tile: int, head_dim: int):
    """(choice 0 per-sequence / 1 per-document, costs [2, cp] int64)."""
    cu = np.ascontiguousarray(cu_seqlens_host, dtype=np.int32)
    costs = np.zeros(2 * cp, dtype=np.int64)
    rc = lib().pva_wlb_choose(cu.ctypes.data_as(ctypes.c_void_p), cu.shape[0] - 1, cp, tile,
                              head_dim, costs.ctypes.data_as(ctypes.c_void_p))
    if rc < 0:
        raise _lib.PvaError("pva_wlb_choose", 1)
    return int(rc), costs.reshape(2, cp)


def debug_withhold_kv_load(enable: bool) -> None:
    """Test hook (see pva_debug_withhold_kv_load): while enabled, one CTA of each
    attention launch (CTA 0 under static dispatch, the one that claimed the
    first unit under dynamic dispatch) waits for a K/V copy that is never
    issued, so its bounded wait expires and worklist_error() reports the site."""
    lib().pva_debug_withhold_kv_load(1 if enable else 0)


def worklist_counts(worklist: torch.Tensor, stream=None) -> dict:
    out = (ctypes.c_int64 * 7)()
    st = lib().pva_worklist_counts(_ptr(worklist), out, _stream(stream))
    names = ("segs", "slices", "units", "runs", "pairs_per_head", "tiles_per_head", "lpt_steps")
    res = dict(zip(names, (int(x) for x in out)))
    res["status"] = int(st)
    return res


# ----------------------------------------------------------------- decoding
_HDR = np.dtype([("i32", "<i4", 20), ("c_tile", "<i8"), ("pair_sum", "<u8"), ("tile_sum", "<u8"),
                 ("off", "<i8", 14)])
_OFF = ("slices", "segs", "units_enum", "keys", "order", "assign", "units", "runs",
        "cta_off", "doc_scan", "dorder", "cls_work", "smask", "total")


def decode_worklist(worklist: torch.Tensor) -> dict:
    """Copy a built worklist to the host and split it into numpy arrays:
    segments, slices, runs and the units.  A static-dispatch worklist gives
    its units in CTA order with the CSR offsets of the CTAs; a dynamic one
    gives them in enumeration (uid) order (cta -1, no offsets) with the
    dispatch order of the uids."""
    raw = worklist.detach().cpu().numpy()
    h = np.frombuffer(raw[:_HDR.itemsize].tobytes(), dtype=_HDR)[0]
    i32 = h["i32"]
    names = ("magic", "version", "error", "num_ctas", "tile_m", "tile_n", "hq", "hkv", "kind",
             "q_tokens", "k_tokens", "num_docs", "cap_slices", "cap_segs", "cap_units",
             "cap_runs", "nslices", "nsegs", "nunits", "nruns")
    hd = {n: int(x) for n, x in zip(names, i32)}
    off = {n: int(x) for n, x in zip(_OFF, h["off"])}
    # after the offsets: lpt_steps, refine_iters, refine_rounds, dispatch_next,
    # dispatch_done, dispatch, dispatch_split, pack_docs
    tail = np.frombuffer(raw[_HDR.itemsize:_HDR.itemsize + 32].tobytes(), dtype="<i4")
    dispatch = tail[5]

    def arr(name, dtype, n, width):
        b = raw[off[name]: off[name] + n * width * np.dtype(dtype).itemsize]
        return np.frombuffer(b.tobytes(), dtype=dtype).reshape(n, width) if width > 1 else \
            np.frombuffer(b.tobytes(), dtype=dtype)

    dynamic = dispatch == DISPATCH_DYNAMIC
    # dynamic dispatch: no per-CTA lists; the units in enumeration (uid) order
    units = arr("units_enum" if dynamic else "units", "<i4", hd["nunits"], 16)
    costs = units[:, 12:14].copy().view("<i8").reshape(-1)
    pairs = units[:, 14:16].copy().view("<i8").reshape(-1)
    return {"header": hd, "pair_sum": int(h["pair_sum"]), "tile_sum": int(h["tile_sum"]),
            "slices": arr("slices", "<i4", hd["nslices"], 8),
            "slice_masks": arr("smask", "<u4", hd["nslices"], 4),
            "pack_docs": int(tail[7]),
            "segs": arr("segs", "<i4", hd["nsegs"], 8),
            "units": units[:, :10].copy(), "unit_ntiles": units[:, 10].copy(),
            "unit_cost": costs, "unit_pairs": pairs,
            "runs": arr("runs", "<i4", hd["nruns"], 4)[:, :3].copy(),
            "cta_off": None if dynamic else arr("cta_off", "<i4", hd["num_ctas"] + 1, 1).copy(),
            "dispatch": int(dispatch), "dispatch_split": int(tail[6]),
            "dispatch_order": arr("dorder", "<i4", hd["nunits"], 1).copy() if dynamic else None}


class PackedAttention:
    """Convenience holder: builds the worklist once for a pack/mask and runs
    the forward on it.  Buffers come from PyTorch; all work is in libpva."""

    def __init__(self, cu_seqlens: Optional[torch.Tensor], mask: MaskDesc,
                 num_q_heads: int, num_kv_heads: int, num_ctas: int = 0,
                 c_tile: Optional[int] = None, head_dim: int = 128):
        self.cu = cu_seqlens
        self.mask = mask
        if c_tile is None:
            c_tile = default_c_tile(head_dim)
        self.params = make_params(num_q_heads, num_kv_heads, num_ctas, c_tile)
        nd = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
        dev = cu_seqlens.device if cu_seqlens is not None else torch.device("cuda")
        self.worklist = alloc_worklist(nd, mask, self.params, dev)

    def plan(self, stream=None) -> None:
        build_worklist(self.cu, self.mask, self.params, self.worklist, stream)

    def forward(self, q, k, v, out=None, lse=None, out_fp32: bool = False, softmax_scale=0.0,
                cta_busy=None, stream=None):
        tq, hq, d = q.shape
        if out is None:
            out = torch.empty((tq, hq, d), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                              device=q.device)
        if lse is None:
            lse = torch.empty((hq, tq), dtype=torch.float32, device=q.device)
        attn_fwd(q, k, v, self.cu, self.mask, self.params, self.worklist, out, lse,
                 softmax_scale, cta_busy, stream)
        return out, lse


def mask_for_workload(w, q_tokens: Optional[int] = None, k_tokens: Optional[int] = None,
                      **kw) -> MaskDesc:
    t = w.total_tokens
    return make_mask(w.mask_kind, q_tokens if q_tokens is not None else t,
                     k_tokens if k_tokens is not None else t, window=w.window,
                     num_prefix_docs=w.num_prefix_docs, **kw)
