"""CPU checks of the C ABI: the library loads, exports every symbol that
include/pva.h declares, and rejects bad arguments on the host before any
device work.  No compute call is made (there is no GPU here)."""
import ctypes
import os
import re

import numpy as np
import pytest

from packed_varlen_attention_cu_gb300 import _lib, api
from packed_varlen_attention_cu_gb300 import build as pva_build
from packed_varlen_attention_cu_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pva.h")


@pytest.fixture(scope="module")
def L():
    pva_build.build()
    return _lib.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pva_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    assert L.pva_status_string(0) == b"ok"
    assert L.pva_status_string(5) == b"device-side wait timed out"
    assert L.pva_version() == 10000


def test_worklist_bytes_bounds(L):
    w = W.zigzag_pack()
    mask = api.mask_for_workload(w)
    p = api.make_params(32, 8, num_ctas=152)
    n = api.worklist_bytes(w.num_docs, mask, p)
    assert 256 < n < 64 << 20
    # invalid: heads not divisible, zero tiles, too many CTAs, bad window
    for bad in (api.make_params(32, 6, num_ctas=152), api.make_params(32, 8, num_ctas=152, tile_m=0),
                api.make_params(32, 8, num_ctas=2048)):
        assert L.pva_worklist_bytes(w.num_docs, ctypes.byref(mask), ctypes.byref(bad)) == 0
    bad_mask = api.make_mask(W.MASK_SLIDING_WINDOW, 10, 10, window=0)
    assert L.pva_worklist_bytes(1, ctypes.byref(bad_mask), ctypes.byref(p)) == 0


def test_overlapping_slices_rejected(L):
    sl = np.array([[0, 10, 0, 0, 10, 0, 1, 0], [5, 10, 0, 0, 10, 0, 1, 0]], dtype=np.int32)
    m = api.make_mask(W.MASK_SLICES, 20, 20, slices=sl)
    p = api.make_params(2, 2, num_ctas=4)
    assert L.pva_worklist_bytes(0, ctypes.byref(m), ctypes.byref(p)) == 0


def test_zigzag_shard_len_matches_oracle(L, oracle_mod):
    w = W.zigzag_pack()
    for cp in (1, 2, 8):
        total = 0
        for r in range(cp):
            n = api.zigzag_shard_len(w.cu_seqlens, cp, r)
            assert n == oracle_mod.zigzag_map(w.cu_seqlens, cp, r)[0].shape[0]
            total += n
        assert total == w.total_tokens
    assert L.pva_zigzag_shard_len(w.cu_seqlens.ctypes.data_as(ctypes.c_void_p), w.num_docs, 2, 2) == -1


def test_host_argument_checks_return_codes(L):
    m = api.make_mask(W.MASK_CAUSAL, 128, 128)
    p = api.make_params(2, 2, num_ctas=4)
    fake = ctypes.c_void_p(256)
    # null mask / params / worklist
    assert L.pva_build_worklist(fake, 1, None, ctypes.byref(p), fake, 1 << 20, None) == 1
    # misaligned worklist buffer
    assert L.pva_build_worklist(fake, 1, ctypes.byref(m), ctypes.byref(p), ctypes.c_void_p(260),
                                1 << 20, None) == 1
    # buffer too small
    assert L.pva_build_worklist(fake, 1, ctypes.byref(m), ctypes.byref(p), fake, 16, None) == 2
    # unsupported head dim / tiles, before any device work
    assert L.pva_attn_fwd(fake, fake, fake, fake, ctypes.byref(m), ctypes.byref(p), 96, fake, fake,
                          0, fake, 0.0, None, None) == 4
    p64 = api.make_params(2, 2, num_ctas=4, tile_m=64)
    assert L.pva_attn_fwd(fake, fake, fake, fake, ctypes.byref(m), ctypes.byref(p64), 64, fake,
                          fake, 0, fake, 0.0, None, None) == 4
    # misaligned q
    assert L.pva_attn_fwd(ctypes.c_void_p(258), fake, fake, fake, ctypes.byref(m), ctypes.byref(p),
                          64, fake, fake, 0, fake, 0.0, None, None) == 1
    # merge: head dim whose rows would straddle warps, bad flag
    assert L.pva_merge_partials(fake, fake, fake, fake, fake, fake, 8, 2, 96, 1, None) == 4
    assert L.pva_merge_partials(fake, fake, fake, fake, fake, fake, 8, 2, 64, 2, None) == 1
    # gather: row bytes not a multiple of 16
    assert L.pva_gather_rows(fake, fake, fake, 4, 24, 4, 0, None) == 1
    # zigzag: rank out of range
    assert L.pva_zigzag_shard(fake, 3, 2, 5, fake, None, None) == 1


def test_sharding_solver_host_checks(L):
    fake = ctypes.c_void_p(256)
    m = api.make_mask(W.MASK_CAUSAL, 128, 128)
    # chunk areas: bad chunk size; rank-local mask kinds are not whole-pack masks
    assert L.pva_chunk_areas(fake, 1, ctypes.byref(m), 0, fake, None) == 1
    mz = api.make_mask(W.MASK_ZIGZAG_PAIR, 64, 64, cp=2, q_rank=0, k_rank=1)
    assert L.pva_chunk_areas(fake, 1, ctypes.byref(mz), 16, fake, None) == 4
    # dispatch: buckets must take whole shares; size limits
    assert L.pva_dispatch_chunks(fake, 10, 4, fake, fake, None) == 1
    assert L.pva_dispatch_chunks(fake, 16384, 8, fake, fake, None) == 4
    assert L.pva_dispatch_chunks(fake, 2048, 2048, fake, fake, None) == 4
    # striped: bad stripe / rank
    assert L.pva_striped_shard_len(100, 4, 4, 1) == -1 and L.pva_striped_shard_len(100, 4, 0, 0) == -1
    assert L.pva_striped_shard(100, 4, 0, 0, fake, None) == 1


@pytest.mark.parametrize("T,cp,stripe", [(131072, 8, 1), (131072, 8, 1024), (1000, 3, 7), (5, 8, 2)])
def test_striped_shard_len_matches_oracle(oracle_mod, T, cp, stripe):
    lens = [api.striped_shard_len(T, cp, r, stripe) for r in range(cp)]
    assert lens == [oracle_mod.striped_map(T, cp, r, stripe).shape[0] for r in range(cp)]
    assert sum(lens) == T


def test_wlb_choose_matches_oracle(oracle_mod):
    packs = [W.zigzag_pack().cu_seqlens, W.cu_seqlens_of([64] * 64),
             W.cu_seqlens_of([256] * 16 + [16384]), W.cu_seqlens_of([8192]),
             W.cu_seqlens_of([70, 5, 300, 129, 1, 200])]
    packs += [W.long_tail_gqa().cu_seqlens[:9] - 0]  # first 8 documents
    for cu in packs:
        for cp, tile, d in ((2, 32, 64), (4, 128, 128), (8, 128, 128)):
            got = api.wlb_choose(cu, cp, tile, d)
            want = oracle_mod.wlb_choose(cu, cp, tile, d)
            assert got[0] == want[0] and np.array_equal(got[1], want[1])


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.lib()
