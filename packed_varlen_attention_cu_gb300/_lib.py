"""ctypes view of ``libpva.so`` (declarations mirror include/pva.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpva.so")

PVA_OK = 0
STATUS_NAMES = {0: "PVA_OK", 1: "PVA_ERR_INVALID_ARG", 2: "PVA_ERR_BUFFER_TOO_SMALL",
                3: "PVA_ERR_CUDA", 4: "PVA_ERR_UNSUPPORTED", 5: "PVA_ERR_TIMEOUT",
                6: "PVA_ERR_DEVICE"}

# Every symbol declared by include/pva.h.
EXPORTS = ("pva_worklist_bytes", "pva_build_worklist", "pva_attn_fwd", "pva_attn_fwd_accumulate",
           "pva_zigzag_shard_len",
           "pva_zigzag_shard", "pva_zigzag_ring_map", "pva_gather_rows", "pva_merge_partials", "pva_worklist_error",
           "pva_worklist_counts", "pva_attn_fwd_noalloc", "pva_noalloc_scratch_bytes",
           "pva_noalloc_error",
           "pva_attn_fwd_host",
           "pva_debug_withhold_kv_load", "pva_chunk_areas", "pva_dispatch_chunks",
           "pva_striped_shard_len", "pva_striped_shard", "pva_wlb_choose",
           "pva_fit_tile_cost",
           "pva_bwd_plan_bytes", "pva_build_bwd_plan", "pva_attn_bwd",
           "pva_status_string", "pva_version")


class Slice(ctypes.Structure):
    _fields_ = [("q_row0", ctypes.c_int32), ("q_len", ctypes.c_int32), ("q_pos0", ctypes.c_int32),
                ("k_row0", ctypes.c_int32), ("k_len", ctypes.c_int32), ("k_pos0", ctypes.c_int32),
                ("type", ctypes.c_int32), ("window", ctypes.c_int32)]


class MaskDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32),
                ("num_prefix_docs", ctypes.c_int32), ("cp", ctypes.c_int32),
                ("q_rank", ctypes.c_int32), ("k_rank", ctypes.c_int32),
                ("slices", ctypes.POINTER(Slice)), ("num_slices", ctypes.c_int32),
                ("q_tokens", ctypes.c_int32), ("k_tokens", ctypes.c_int32),
                ("ring_step", ctypes.c_int32)]


class WorklistParams(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("num_ctas", ctypes.c_int32), ("refine_iters", ctypes.c_int32),
                ("c_tile", ctypes.c_int64), ("dispatch", ctypes.c_int32),
                ("pack_docs", ctypes.c_int32)]


class PvaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                "g.build()\"` (needs nvcc); there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        MP, WP = ctypes.POINTER(MaskDesc), ctypes.POINTER(WorklistParams)
        L.pva_worklist_bytes.restype = sz
        L.pva_worklist_bytes.argtypes = [i32, MP, WP]
        L.pva_build_worklist.restype = ctypes.c_int
        L.pva_build_worklist.argtypes = [P, i32, MP, WP, P, sz, P]
        L.pva_attn_fwd.restype = ctypes.c_int
        L.pva_attn_fwd.argtypes = [P, P, P, P, MP, WP, i32, P, P, i32, P, ctypes.c_float, P, P]
        L.pva_attn_fwd_accumulate.restype = ctypes.c_int
        L.pva_attn_fwd_accumulate.argtypes = [P, P, P, P, MP, WP, i32, P, P, P, ctypes.c_float, P,
                                              P]
        L.pva_zigzag_shard_len.restype = i32
        L.pva_zigzag_shard_len.argtypes = [P, i32, i32, i32]
        L.pva_zigzag_shard.restype = ctypes.c_int
        L.pva_zigzag_shard.argtypes = [P, i32, i32, i32, P, P, P]
        L.pva_zigzag_ring_map.restype = ctypes.c_int
        L.pva_zigzag_ring_map.argtypes = [P, i32, i32, P, P]
        L.pva_gather_rows.restype = ctypes.c_int
        L.pva_gather_rows.argtypes = [P, P, P, i64, i64, i64, i32, P]
        L.pva_merge_partials.restype = ctypes.c_int
        L.pva_merge_partials.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, P]
        L.pva_worklist_error.restype = ctypes.c_int
        L.pva_worklist_error.argtypes = [P, ctypes.POINTER(i32), P]
        L.pva_worklist_counts.restype = ctypes.c_int
        L.pva_worklist_counts.argtypes = [P, ctypes.POINTER(i64), P]
        L.pva_attn_fwd_noalloc.restype = ctypes.c_int
        L.pva_attn_fwd_noalloc.argtypes = [P, P, P, P, i32, MP, WP, i32, P, i32, P,
                                           ctypes.c_float, P]
        L.pva_noalloc_scratch_bytes.restype = sz
        L.pva_noalloc_scratch_bytes.argtypes = []
        L.pva_noalloc_error.restype = ctypes.c_int
        L.pva_noalloc_error.argtypes = [ctypes.POINTER(i32), P]
        L.pva_attn_fwd_host.restype = ctypes.c_int
        L.pva_attn_fwd_host.argtypes = [P, P, P, P, i32, MP, WP, i32, P, P, ctypes.c_float,
                                        P, P, P, P, P, sz, P, P, P]
        L.pva_chunk_areas.restype = ctypes.c_int
        L.pva_chunk_areas.argtypes = [P, i32, MP, i32, P, P]
        L.pva_dispatch_chunks.restype = ctypes.c_int
        L.pva_dispatch_chunks.argtypes = [P, i32, i32, P, P, P]
        L.pva_striped_shard_len.restype = i32
        L.pva_striped_shard_len.argtypes = [i32, i32, i32, i32]
        L.pva_striped_shard.restype = ctypes.c_int
        L.pva_striped_shard.argtypes = [i32, i32, i32, i32, P, P]
        L.pva_wlb_choose.restype = i32
        L.pva_wlb_choose.argtypes = [P, i32, i32, i32, i32, P]
        L.pva_fit_tile_cost.restype = ctypes.c_int
        L.pva_fit_tile_cost.argtypes = [P, P, i32, P, P, P]
        L.pva_bwd_plan_bytes.restype = sz
        L.pva_bwd_plan_bytes.argtypes = [i32, MP, WP]
        L.pva_build_bwd_plan.restype = ctypes.c_int
        L.pva_build_bwd_plan.argtypes = [P, i32, MP, WP, P, sz, P]
        L.pva_attn_bwd.restype = ctypes.c_int
        L.pva_attn_bwd.argtypes = [P, P, P, P, P, P, P, i32, MP, WP, i32, P, P, P, P, P, i32,
                                   ctypes.c_float, P]
        L.pva_debug_withhold_kv_load.restype = None
        L.pva_debug_withhold_kv_load.argtypes = [i32]
        L.pva_status_string.restype = ctypes.c_char_p
        L.pva_status_string.argtypes = [ctypes.c_int]
        L.pva_version.restype = i32
        L.pva_version.argtypes = []
        _lib = L
    return _lib


def check(fn: str, status: int) -> None:
    if status != PVA_OK:
        raise PvaError(fn, status)
