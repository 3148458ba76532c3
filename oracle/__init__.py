"""Python view of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check
and by the benchmark's CPU-baseline leg, never by the product path.  It
shares no code with the CUDA library.

Functions mirror the C entry points and take/return numpy arrays.  bf16
tensors are passed as their raw uint16 bit patterns; the C side widens them
exactly to fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

(MASK_CAUSAL, MASK_SLIDING_WINDOW, MASK_SHARED_QUESTION, MASK_ZIGZAG_PAIR, MASK_SLICES,
 MASK_ZIGZAG_STEP) = range(6)
SLICE_FULL, SLICE_CAUSAL, SLICE_INV_CAUSAL, SLICE_BI_CAUSAL = 0, 1, 2, 3


def compile_oracle(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2, OpenMP) if missing or stale."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Mask(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32),
                ("num_prefix", ctypes.c_int32), ("cp", ctypes.c_int32),
                ("q_rank", ctypes.c_int32), ("k_rank", ctypes.c_int32),
                ("slices", ctypes.POINTER(ctypes.c_int32)), ("num_slices", ctypes.c_int32),
                ("ring_step", ctypes.c_int32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(compile_oracle())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        _lib.or_num_threads.restype = i32
        _lib.or_zigzag_map.restype = i32
        _lib.or_zigzag_map.argtypes = [P, i32, i32, i32, P, P]
        _lib.or_attention.restype = ctypes.c_int
        _lib.or_attention.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, i32,
                                      ctypes.POINTER(_Mask), ctypes.c_double, P, i64, i32, P, P]
        _lib.or_attention_bwd.restype = ctypes.c_int
        _lib.or_attention_bwd.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, i32,
                                          ctypes.POINTER(_Mask), ctypes.c_double, P, P, P]
        _lib.or_attention_bwd_jobs.restype = ctypes.c_int
        _lib.or_attention_bwd_jobs.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, i32,
                                               ctypes.POINTER(_Mask), ctypes.c_double, P, i64,
                                               P, i64, P, P, P]
        _lib.or_pair_count.restype = i64
        _lib.or_pair_count.argtypes = [i32, i32, P, i32, ctypes.POINTER(_Mask), i32]
        _lib.or_allowed_matrix.restype = ctypes.c_int
        _lib.or_allowed_matrix.argtypes = [i32, i32, P, i32, ctypes.POINTER(_Mask), P]
        _lib.or_merge.restype = None
        _lib.or_merge.argtypes = [P, P, P, P, P, P, i64, i32, i32]
        _lib.or_lpt.restype = ctypes.c_int
        _lib.or_lpt.argtypes = [P, i64, i32, P, P, P]
        _lib.or_chunk_areas.restype = ctypes.c_int
        _lib.or_chunk_areas.argtypes = [i32, P, i32, ctypes.POINTER(_Mask), i32, P]
        _lib.or_dispatch_minheap.restype = ctypes.c_int
        _lib.or_dispatch_minheap.argtypes = [P, i32, i32, P, P]
        _lib.or_striped_map.restype = i32
        _lib.or_striped_map.argtypes = [i32, i32, i32, i32, P]
        _lib.or_wlb_choose.restype = ctypes.c_int
        _lib.or_wlb_choose.argtypes = [P, i32, i32, i32, i32, P]
        _lib.or_worklist.restype = ctypes.c_int
        _lib.or_worklist.argtypes = [P, i32, ctypes.POINTER(_Mask), i32, i32, i32, i32, i32,
                                     i64, i32, i32, P, P, P, P, P, P, P, P, P]
        _lib.or_refine_move_swap.restype = ctypes.c_int
        _lib.or_refine_move_swap.argtypes = [P, i64, i32, P, P, i32]
        _lib.or_fit_tile_cost.restype = i64
        _lib.or_fit_tile_cost.argtypes = [P, P, P, i32, P]
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Mask:
    """Mask description understood by the oracle."""

    def __init__(self, kind: int = MASK_CAUSAL, window: int = 0, num_prefix: int = 0,
                 cp: int = 0, q_rank: int = 0, k_rank: int = 0,
                 slices: Optional[np.ndarray] = None, ring_step: int = 0):
        self.kind, self.window, self.num_prefix = kind, window, num_prefix
        self.cp, self.q_rank, self.k_rank = cp, q_rank, k_rank
        self.ring_step = ring_step
        self.slices = None if slices is None else np.ascontiguousarray(slices, dtype=np.int32).reshape(-1, 8)

    def c(self) -> _Mask:
        m = _Mask(self.kind, self.window, self.num_prefix, self.cp, self.q_rank, self.k_rank,
                  None, 0, self.ring_step)
        if self.slices is not None:
            m.slices = self.slices.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
            m.num_slices = self.slices.shape[0]
        return m


def num_threads() -> int:
    return int(lib().or_num_threads())


def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor (any device)."""
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def ring_map(cu: np.ndarray, cp: int) -> np.ndarray:
    """Ring order of all zigzag shards: the maps of ranks 0..cp-1 concatenated."""
    return np.concatenate([zigzag_map(cu, cp, r)[0] for r in range(cp)]).astype(np.int32)


def zigzag_map(cu: np.ndarray, cp: int, rank: int):
    """(gather map [T_r] int32, chunk table [ndocs, 2, 4]) for one rank."""
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    nd = cu.shape[0] - 1
    n = lib().or_zigzag_map(_ptr(cu), nd, cp, rank, None, None)
    if n < 0:
        raise ValueError("bad zigzag arguments")
    m = np.zeros(max(n, 1), dtype=np.int32)
    table = np.zeros((max(nd, 1), 2, 4), dtype=np.int32)
    lib().or_zigzag_map(_ptr(cu), nd, cp, rank, _ptr(m), _ptr(table))
    return m[:n], table[:nd]


def attention(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, cu: np.ndarray,
              mask: Mask, scale: Optional[float] = None, jobs: Optional[np.ndarray] = None,
              brute: bool = False):
    """fp64 attention from bf16 bit patterns.

    q_bits [Tq, Hq, d], k_bits/v_bits [Tk, Hkv, d] (uint16).  Returns
    (out, lse): all rows -> out [Tq, Hq, d], lse [Hq, Tq]; with ``jobs``
    ((row, head) int32 [n, 2]) -> out [n, d], lse [n].
    """
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    Tq, Hq, d = q_bits.shape
    Tk, Hkv, _ = k_bits.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if jobs is None:
        out = np.zeros((Tq, Hq, d), dtype=np.float64)
        lse = np.zeros((Hq, Tq), dtype=np.float64)
        nj = 0
    else:
        jobs = np.ascontiguousarray(jobs, dtype=np.int32).reshape(-1, 2)
        nj = jobs.shape[0]
        out = np.zeros((nj, d), dtype=np.float64)
        lse = np.zeros((nj,), dtype=np.float64)
    m = mask.c()
    rc = lib().or_attention(_ptr(q_bits), _ptr(k_bits), _ptr(v_bits), Tq, Tk, Hq, Hkv, d,
                            _ptr(cu), cu.shape[0] - 1, ctypes.byref(m), float(scale),
                            _ptr(jobs), nj, 1 if brute else 0, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"or_attention failed ({rc})")
    return out, lse


def attention_bwd(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray,
                  do_bits: np.ndarray, cu: np.ndarray, mask: Mask, scale: Optional[float] = None):
    """fp64 gradients (dq [Tq, Hq, d], dk, dv [Tk, Hkv, d]) of attention with
    output gradient dO, from bf16 bit patterns.  Brute force: O(Tq Tk Hq d)."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    do_bits = np.ascontiguousarray(do_bits, dtype=np.uint16)
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    Tq, Hq, d = q_bits.shape
    Tk, Hkv, _ = k_bits.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros((Tq, Hq, d), dtype=np.float64)
    dk = np.zeros((Tk, Hkv, d), dtype=np.float64)
    dv = np.zeros((Tk, Hkv, d), dtype=np.float64)
    m = mask.c()
    rc = lib().or_attention_bwd(_ptr(q_bits), _ptr(k_bits), _ptr(v_bits), _ptr(do_bits), Tq, Tk,
                                Hq, Hkv, d, _ptr(cu), cu.shape[0] - 1, ctypes.byref(m),
                                float(scale), _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError(f"or_attention_bwd failed ({rc})")
    return dq, dk, dv


def attention_bwd_jobs(q_bits, k_bits, v_bits, do_bits, cu, mask: Mask, qjobs, kjobs,
                       scale: Optional[float] = None):
    """Sampled gradients: dq [nq, d] of (row, head) jobs, dk and dv [nk, d] of
    (key, kv head) jobs, each by definition (bf16 bit patterns in)."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    do_bits = np.ascontiguousarray(do_bits, dtype=np.uint16)
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    qj = np.ascontiguousarray(qjobs, dtype=np.int32).reshape(-1, 2)
    kj = np.ascontiguousarray(kjobs, dtype=np.int32).reshape(-1, 2)
    Tq, Hq, d = q_bits.shape
    Tk, Hkv, _ = k_bits.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros((max(len(qj), 1), d))
    dk = np.zeros((max(len(kj), 1), d))
    dv = np.zeros((max(len(kj), 1), d))
    m = mask.c()
    rc = lib().or_attention_bwd_jobs(_ptr(q_bits), _ptr(k_bits), _ptr(v_bits), _ptr(do_bits), Tq,
                                     Tk, Hq, Hkv, d, _ptr(cu), cu.shape[0] - 1, ctypes.byref(m),
                                     float(scale), _ptr(qj), len(qj), _ptr(kj), len(kj), _ptr(dq),
                                     _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError(f"or_attention_bwd_jobs failed ({rc})")
    return dq[:len(qj)], dk[:len(kj)], dv[:len(kj)]


def pair_count(cu: np.ndarray, mask: Mask, Tq: Optional[int] = None, Tk: Optional[int] = None,
               brute: bool = False) -> int:
    """Allowed (q, k) pairs per head."""
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    T = int(cu[-1])
    Tq = T if Tq is None else Tq
    Tk = T if Tk is None else Tk
    m = mask.c()
    r = lib().or_pair_count(Tq, Tk, _ptr(cu), cu.shape[0] - 1, ctypes.byref(m), 1 if brute else 0)
    if r < 0:
        raise ValueError("or_pair_count failed")
    return int(r)


def allowed_matrix(cu: np.ndarray, mask: Mask, Tq: Optional[int] = None,
                   Tk: Optional[int] = None) -> np.ndarray:
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    T = int(cu[-1])
    Tq = T if Tq is None else Tq
    Tk = T if Tk is None else Tk
    out = np.zeros((Tq, Tk), dtype=np.uint8)
    m = mask.c()
    if lib().or_allowed_matrix(Tq, Tk, _ptr(cu), cu.shape[0] - 1, ctypes.byref(m), _ptr(out)) != 0:
        raise ValueError("or_allowed_matrix failed")
    return out.astype(bool)


def merge(oa, la, ob, lb):
    """fp64 online-softmax merge; O [tokens, heads, d], lse [heads, tokens]."""
    oa = np.ascontiguousarray(oa, dtype=np.float64)
    ob = np.ascontiguousarray(ob, dtype=np.float64)
    la = np.ascontiguousarray(la, dtype=np.float64)
    lb = np.ascontiguousarray(lb, dtype=np.float64)
    t, h, d = oa.shape
    o = np.zeros_like(oa)
    l = np.zeros_like(la)
    lib().or_merge(_ptr(oa), _ptr(la), _ptr(ob), _ptr(lb), _ptr(o), _ptr(l), t, h, d)
    return o, l


def lpt(cost: Sequence[int], bins: int):
    """LPT: (assign [n] bin per item, order [n] items in assignment order, loads [bins])."""
    c = np.ascontiguousarray(np.asarray(cost, dtype=np.int64))
    n = c.shape[0]
    assign = np.zeros(max(n, 1), dtype=np.int32)
    order = np.zeros(max(n, 1), dtype=np.int64)
    loads = np.zeros(bins, dtype=np.int64)
    if lib().or_lpt(_ptr(c), n, bins, _ptr(assign), _ptr(order), _ptr(loads)) != 0:
        raise ValueError("or_lpt failed")
    return assign[:n], order[:n], loads


def dispatch_order(cost_by_uid: Sequence[int], num_ctas: int) -> np.ndarray:
    """Run-time dispatch order of a worklist's units (uids), for CTAs that claim
    their next unit when they run out of work.  It follows the LPT rule
    ("数据并行负载均衡" §4.4: largest cost first, each to whichever worker is
    least loaded) over power-of-two cost classes k = floor(log2(max(cost, 1))):
    classes above a split class go first, in decreasing class, enumeration
    order (uid) inside a class; the split class and all below it follow in
    exact LPT order (cost desc, uid asc).  The split is the highest non-empty
    class k whose units the work below it could not absorb, i.e. the work of
    the classes under k is below num_ctas * 2^(k+1) (capped at 38).  Plain
    Python: bit lengths, sums and sorts."""
    cost = [int(c) for c in cost_by_uid]
    classes = [max(c, 1).bit_length() - 1 for c in cost]
    work = {}
    for c, k in zip(cost, classes):
        work[k] = work.get(k, 0) + c
    split = 0
    for k in sorted(work, reverse=True):
        below = sum(wk for kk, wk in work.items() if kk < k)
        if below < num_ctas * 2 ** (k + 1):
            split = min(k, 38)
            break
    upper = sorted((u for u in range(len(cost)) if classes[u] > split),
                   key=lambda u: (-classes[u], u))
    lower = sorted((u for u in range(len(cost)) if classes[u] <= split),
                   key=lambda u: (-cost[u], u))
    return np.asarray(upper + lower, dtype=np.int32)


UNIT_FIELDS = ("uid", "seg", "t0", "t1", "h0", "h1", "kvh", "run_begin", "run_count", "cta")


def worklist(cu: np.ndarray, mask: Mask, tile_m: int, tile_n: int, hq: int, hkv: int,
             num_ctas: int, c_tile: int = 0, refine_iters: int = 0, pack_docs: int = 0) -> dict:
    """Worklist of the method (segments, slices, units in CTA order, runs, CSR).
    pack_docs: short documents share tiles (packed slices, type 4, with the rows
    that start a document in "slice_masks" [n, 4] uint32)."""
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    nd = cu.shape[0] - 1
    counts = np.zeros(5, dtype=np.int64)
    m = mask.c()
    L = lib()
    rc = L.or_worklist(_ptr(cu), nd, ctypes.byref(m), tile_m, tile_n, hq, hkv, num_ctas,
                       int(c_tile), int(refine_iters), int(pack_docs), _ptr(counts), None, None,
                       None, None, None, None, None, None)
    if rc != 0:
        raise ValueError(f"or_worklist failed ({rc})")
    nseg, nsl, nu, nr = (int(x) for x in counts[:4])
    slices = np.zeros((max(nsl, 1), 8), dtype=np.int32)
    smasks = np.zeros((max(nsl, 1), 4), dtype=np.uint32)
    segs = np.zeros((max(nseg, 1), 5), dtype=np.int32)
    units = np.zeros((max(nu, 1), 10), dtype=np.int32)
    cost = np.zeros(max(nu, 1), dtype=np.int64)
    pairs = np.zeros(max(nu, 1), dtype=np.int64)
    runs = np.zeros((max(nr, 1), 3), dtype=np.int32)
    off = np.zeros(num_ctas + 1, dtype=np.int32)
    rc = L.or_worklist(_ptr(cu), nd, ctypes.byref(m), tile_m, tile_n, hq, hkv, num_ctas,
                       int(c_tile), int(refine_iters), int(pack_docs), _ptr(counts),
                       _ptr(slices), _ptr(smasks), _ptr(segs), _ptr(units),
                       _ptr(cost), _ptr(pairs), _ptr(runs), _ptr(off))
    if rc != 0:
        raise ValueError(f"or_worklist failed ({rc})")
    return {"slices": slices[:nsl], "slice_masks": smasks[:nsl], "segs": segs[:nseg],
            "units": units[:nu],
            "unit_cost": cost[:nu], "unit_pairs": pairs[:nu], "runs": runs[:nr],
            "cta_off": off, "pairs_per_head": int(counts[4])}


# ----------------------------------------------------------- dispatch / sharding
def chunk_areas(cu: np.ndarray, mask: Mask, chunk_size: int) -> np.ndarray:
    """Allowed pairs of every chunk of chunk_size query rows ("03" §4.4)."""
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    T = int(cu[-1])
    n = (T + chunk_size - 1) // chunk_size
    areas = np.zeros(max(n, 1), dtype=np.int64)
    m = mask.c()
    rc = lib().or_chunk_areas(T, _ptr(cu), cu.shape[0] - 1, ctypes.byref(m), chunk_size,
                              _ptr(areas))
    if rc < 0:
        raise ValueError("or_chunk_areas failed")
    return areas[:n]


def dispatch_minheap(areas: Sequence[int], cp: int):
    """Greedy min-heap dispatch ("03" §4.4): (bucket [n], loads [cp])."""
    a = np.ascontiguousarray(np.asarray(areas, dtype=np.int64))
    n = a.shape[0]
    bucket = np.zeros(max(n, 1), dtype=np.int32)
    loads = np.zeros(cp, dtype=np.int64)
    if lib().or_dispatch_minheap(_ptr(a), n, cp, _ptr(bucket), _ptr(loads)) != 0:
        raise ValueError("or_dispatch_minheap failed")
    return bucket[:n], loads


def striped_map(T: int, cp: int, rank: int, stripe: int) -> np.ndarray:
    """Tokens of `rank` under striped sharding ("03" §4.2), in order."""
    n = lib().or_striped_map(T, cp, rank, stripe, None)
    if n < 0:
        raise ValueError("bad striped arguments")
    out = np.zeros(max(n, 1), dtype=np.int32)
    lib().or_striped_map(T, cp, rank, stripe, _ptr(out))
    return out[:n]


def wlb_choose(cu: np.ndarray, cp: int, tile: int, d: int):
    """WLB-LLM per-seq vs per-doc choice ("03" §4.3): (choice, costs [2, cp])."""
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    costs = np.zeros(2 * cp, dtype=np.int64)
    rc = lib().or_wlb_choose(_ptr(cu), cu.shape[0] - 1, cp, tile, d, _ptr(costs))
    if rc < 0:
        raise ValueError("or_wlb_choose failed")
    return int(rc), costs.reshape(2, cp)


def refine_move_swap(cost: Sequence[int], assign: Sequence[int], bins: int, max_iters: int):
    """Move/swap refinement after LPT ("数据并行负载均衡" §4.4 phase 2):
    (assign [n], loads [bins], rounds applied)."""
    c = np.ascontiguousarray(np.asarray(cost, dtype=np.int64))
    a = np.array(assign, dtype=np.int32)
    loads = np.zeros(bins, dtype=np.int64)
    np.add.at(loads, a, c)
    k = lib().or_refine_move_swap(_ptr(c), c.shape[0], bins, _ptr(a), _ptr(loads), max_iters)
    return a, loads, int(k)


def fit_tile_cost(P: Sequence[int], U: Sequence[int], t: Sequence[float]):
    """Per-tile cost from per-bin times ("数据并行负载均衡" §4.2):
    (c_tile, (a, c)) with t ~ a P + c U, a, c >= 0; c_tile = -1 if degenerate."""
    p = np.ascontiguousarray(np.asarray(P, dtype=np.int64))
    u = np.ascontiguousarray(np.asarray(U, dtype=np.int64))
    tt = np.ascontiguousarray(np.asarray(t, dtype=np.float64))
    coef = np.zeros(2, dtype=np.float64)
    ct = lib().or_fit_tile_cost(_ptr(p), _ptr(u), _ptr(tt), p.shape[0], _ptr(coef))
    return int(ct), tuple(float(x) for x in coef)
